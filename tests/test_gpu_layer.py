"""GPU parity of one MoE layer against the fp64 oracle, through the C ABI.

Routing arrays must match bit for bit (inputs drawn so every token's 8th/9th
logit gap is >= 1e-3); top-k weights within 1e-5; outputs within
max|y_gpu - y_oracle| <= 2e-2 * rms(y_oracle).
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


class Case:
    """One layer on the GPU plus its host copies for the oracle."""

    def __init__(self, w: synth.Workload, layer: int = 0, gap: bool = True):
        self.w = w
        sh = w.shape
        self.L = stack.make_layer(w, layer, "cuda")
        self.x = synth.tokens_x(w, "cuda")
        if gap:
            parity.enforce_gap(w, self.x, self.L.router_w, self.L.router_bias, sh.top_k)
        self.xh = parity.bits(self.x)
        self.wr = parity.bits(self.L.router_w)
        self.rb = None if self.L.router_bias is None else self.L.router_bias.cpu().numpy()
        self.routed = parity.host_set(self.L.routed)
        self.shared = parity.host_set(self.L.shared) if self.L.shared is not None else None

    def oracle_route(self):
        orc = oracle.get()
        sh = self.w.shape
        logits = orc.router_logits(self.xh, self.wr, self.rb)
        idx, w, gap = orc.topk(logits, sh.top_k)
        maps = orc.route_maps(idx, sh.num_experts, 128)
        return logits, idx, w, gap, maps

    def oracle_layer(self, rows=None):
        sh = self.w.shape
        return oracle.get().moe_rows(self.xh, self.wr, self.rb, self.routed, self.shared,
                                     sh.top_k, sh.group_size, rows=rows, nthreads=NTHREADS)


def make_plan(w: synth.Workload, gemm_path=0, max_tokens=None):
    """A plan for the workload's shape (capacity: its T, or max_tokens)."""
    sh = w.shape
    d = bg.plan_desc(sh.hidden, sh.inter, sh.num_experts, sh.top_k, sh.group_size,
                     int(sh.has_shared), max_tokens or w.tokens, 128, gemm_path)
    return bg.moe_plan_create(d, 0)


WL = synth.standard_workloads()
SMALL = synth.MoEShape(hidden=256, inter=256, num_experts=16, top_k=4)


@pytest.mark.parametrize("name", ["t128_uniform", "t512_zipf", "t2048_uniform", "t2048_zipf",
                                  "prefill_t4096_l40_zipf", "decode_t1_l40", "decode_t8_l40"])
def test_route_bit_exact(name):
    """Routing against the oracle; the decode sizes exercise the router's
    GEMV path for batches of at most 16 tokens."""
    w = WL[name]
    c = Case(w)
    plan = make_plan(w)
    try:
        r = bg.moe_route(plan, c.x, w.tokens, c.L.router_w, c.L.router_bias)
        g = parity.routing_to_numpy(r, w.tokens, w.shape.top_k, w.shape.num_experts)
        logits, idx, wts, gap, maps = c.oracle_route()
        assert gap.min() >= parity.GAP_MIN
        np.testing.assert_allclose(g["logits"], logits, rtol=0, atol=1e-4)
        assert np.array_equal(g["topk_idx"], idx)
        assert np.abs(g["topk_w"] - wts).max() <= parity.W_TOL
        assert np.abs(g["topk_w"].sum(axis=1) - 1).max() <= 1e-6
        for key in ("counts", "offsets", "tile_offsets", "perm", "inv", "block_map"):
            assert np.array_equal(g[key], maps[key]), key
        assert g["num_tiles"] == maps["num_tiles"]
        check_route_invariants(g, g["topk_idx"], w.shape.num_experts, 128)
        if w.routing == "zipf":
            assert g["counts"].max() > 4 * g["counts"].mean()    # skewed groups
            assert (g["counts"] == 0).any()
    finally:
        bg.moe_plan_destroy(plan)


def run_layer(c: Case, plan: int):
    w = c.w
    y = torch.empty(c.x.shape, dtype=torch.float32, device="cuda")
    bg.moe_forward_layer(plan, c.x, w.tokens, c.L.router_w, c.L.router_bias, c.L.routed_c,
                         c.L.shared_c, y)
    torch.cuda.synchronize()
    assert bg.moe_get_error(plan) == 0
    return y


# gemm_path 1 and 0 (auto) take the single-SM tensor-core kernel, 3 the
# SM-pair one, 2 the small-M kernel
LAYER_CASES = [
    ("t128_uniform", 1), ("t128_uniform", 2), ("t128_uniform", 3), ("t512_zipf", 0),
    ("t512_zipf", 2), ("t512_zipf", 3),
]


@pytest.mark.parametrize("name,path", LAYER_CASES)
def test_layer_parity_full(name, path):
    w = WL[name]
    c = Case(w)
    plan = make_plan(w, path)
    try:
        y = run_layer(c, plan)
        assert bg.moe_last_gemm_path(plan) == {0: 1, 3: 4}.get(path, path)
        orc = c.oracle_layer()
        parity.check_y(y.double().cpu().numpy(), orc["y"])
    finally:
        bg.moe_plan_destroy(plan)


@pytest.mark.parametrize("name", ["t2048_uniform", "t2048_zipf", "prefill_t4096_l40_zipf"])
def test_layer_parity_all_rows(name):
    """Every output row of a full-size layer against the oracle (layer 0 of
    the 40-layer stack for the 4096-token workload), so every tile of every
    expert -- full, partial and the hot experts' many -- is compared; for the
    default path and for the SM-pair tensor-core path (256-row tiles)."""
    w = WL[name]
    c = Case(w)
    plan = make_plan(w)
    plan2 = make_plan(w, 3)
    try:
        y = run_layer(c, plan)
        y2 = run_layer(c, plan2)
        assert bg.moe_last_gemm_path(plan2) == 4
        orc = c.oracle_layer()
        r = bg.moe_route(plan, c.x, w.tokens, c.L.router_w, c.L.router_bias)
        g = parity.routing_to_numpy(r, w.tokens, w.shape.top_k, w.shape.num_experts)
        assert np.array_equal(g["topk_idx"], orc["topk_idx"])
        parity.check_y(y.double().cpu().numpy(), orc["y"])
        parity.check_y(y2.double().cpu().numpy(), orc["y"])
    finally:
        bg.moe_plan_destroy(plan)
        bg.moe_plan_destroy(plan2)


def last_round_pieces(num_tiles: int, T: int, sh, num_sms: int):
    """How the tensor-core GEMM deals the last round of units, per pass
    (gate/up, down): units = (routed tiles + shared tiles) x weight blocks;
    the grid is min(SMs, the host's unit bound); r units are left after the
    full rounds, each cut into two K halves when r <= grid / 2."""
    sh_tiles = -(-T // 128) if sh.has_shared else 0
    bound = min(-(-T * sh.top_k // 128) + sh.num_experts, T * sh.top_k)
    out = []
    for nblk, K in ((sh.inter // 128, sh.hidden), (sh.hidden // 256, sh.inter)):
        units = (num_tiles + sh_tiles) * nblk
        G = max(1, min(num_sms, (bound + sh_tiles) * nblk))
        r = units % G
        out.append(2 if r and G // r >= 2 and K // 256 >= 2 else 1)
    return out


@pytest.mark.parametrize("name,tokens", [("t2048_zipf", 0), ("prefill_t4096_l40_zipf", 0),
                                         ("t2048_zipf", 700)])
def test_split_last_round(name, tokens):
    """The split of the GEMM's last round of units (each left-over unit summed
    over two K halves on two SMs, which the second to finish adds): the
    workload's own routing is checked to split the gate/up pass, every output
    row with the split on and off is compared with the oracle, and two runs
    with the split give the same bits (the SM that adds the halves changes
    from run to run; their sum does not). At 700 tokens both passes split and
    the last units, always in the split round, are the shared expert's
    partial tile of 60 rows."""
    w = WL[name] if not tokens else dataclasses.replace(WL[name], tokens=tokens)
    sh = w.shape
    c = Case(w)
    plan = make_plan(w)
    try:
        r = bg.moe_route(plan, c.x, w.tokens, c.L.router_w, c.L.router_bias)
        g = parity.routing_to_numpy(r, w.tokens, sh.top_k, sh.num_experts)
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        pieces = last_round_pieces(int(g["num_tiles"]), w.tokens, sh, sms)
        assert pieces[0] > 1, pieces
        if w.tokens % 128:
            assert pieces[1] > 1, pieces
        bg.moe_set_tail_split(plan, True)
        y1 = run_layer(c, plan).clone()
        y2 = run_layer(c, plan).clone()
        assert np.array_equal(y1.cpu().numpy(), y2.cpu().numpy())
        bg.moe_set_tail_split(plan, False)
        y0 = run_layer(c, plan)
        assert bg.moe_last_gemm_path(plan) == 1
        orc = c.oracle_layer()
        parity.check_y(y1.double().cpu().numpy(), orc["y"])
        parity.check_y(y0.double().cpu().numpy(), orc["y"])
        assert not np.array_equal(y1.cpu().numpy(), y0.cpu().numpy())   # the split ran
    finally:
        bg.moe_plan_destroy(plan)


def _tie_bias(kind: str, E: int) -> np.ndarray:
    """Router biases that make every token's logits exactly these values
    (the router weight is zero): ties, signed zeros and NaNs."""
    nan = np.float32("nan")
    b = np.full(E, -1.0, np.float32)
    if kind == "ties":          # ten experts tied at 0.5; the top 8 are the lowest indices
        b[[3, 9, 17, 40, 41, 100, 130, 200, 201, E - 1]] = 0.5
        b[[5, 6]] = 0.25
    elif kind == "signed_zero":  # +0 and -0 tie at the top
        b[:] = -2.0
        b[[2, 4, 8, 16, 32, 64, 128, E - 3, E - 2, E - 1]] = [0.0, -0.0] * 5
    elif kind == "nan":          # four finite experts, the rest NaN: four picks of weight 0
        b[:] = nan
        b[[7, 11, 13, 250]] = 1.0
    elif kind == "all_nan":
        b[:] = nan
    return b


@pytest.mark.parametrize("T", [5, 100])
@pytest.mark.parametrize("kind", ["ties", "signed_zero", "nan", "all_nan"])
def test_routing_ties_nan_signed_zero(T, kind):
    """Routing edge cases on the GPU against the oracle's top-k: exact ties
    (the lower expert index wins, in selection and slot order), -0 tying
    with +0, and NaN logits ranking as -infinity with weight zero. The router
    weight is zero, so each logit is exactly its bias; the chosen weights are
    exact binary fractions (or 0, or NaN), so they compare bit for bit. T = 5
    takes the one-launch decode routing, T = 100 the cooperative one; the
    allocation-free entry point (separate launches) is checked too. The
    weights are compared bit for bit after rounding the oracle's fp64
    weights to the FP32 the GPU stores (the fp64 renormalisation itself can
    round in the last place: a sum of eight equal terms)."""
    sh = synth.MoEShape()
    E, k = sh.num_experts, sh.top_k
    w = synth.Workload(f"ties{T}", T, 1, "uniform", seed=901 + T, shape=sh)
    x = synth.tokens_x(w, "cuda")
    wr = torch.zeros((sh.hidden, E), dtype=torch.bfloat16, device="cuda")
    bias = _tie_bias(kind, E)
    rb = torch.from_numpy(bias).cuda()
    orc = oracle.get()
    logits = orc.router_logits(parity.bits(x), parity.bits(wr), bias)
    idx, wts, _ = orc.topk(logits, k)
    plan = make_plan(w, max_tokens=T)
    try:
        outs = [parity.routing_to_numpy(bg.moe_route(plan, x, T, wr, rb), T, k, E)]
        bufs, r = parity.caller_routing_buffers(T, k, E)
        bg.moe_route_noalloc(x, T, sh.hidden, wr, rb, E, k, r)
        outs.append(parity.routing_to_numpy(r, T, k, E))
        assert bg.moe_route_noalloc_get_error() == 0
        assert bg.moe_get_error(plan) == 0
        for g in outs:
            assert np.array_equal(g["topk_idx"], idx)
            gw = g["topk_w"]
            w32 = wts.astype(np.float32)
            assert np.array_equal(np.isnan(gw), np.isnan(w32))
            fin = ~np.isnan(w32)
            assert np.array_equal(gw[fin].view(np.uint32), w32[fin].view(np.uint32))
            maps = orc.route_maps(g["topk_idx"], E, 128)
            for key in ("counts", "offsets", "tile_offsets", "perm", "inv", "block_map"):
                assert np.array_equal(g[key], maps[key]), key
        if kind == "ties":
            assert idx[0].tolist() == [3, 9, 17, 40, 41, 100, 130, 200]
            assert np.all(np.abs(wts - 0.125) <= 1e-15)
        elif kind == "nan":
            assert idx[0].tolist() == [7, 11, 13, 250, 0, 1, 2, 3]
            assert np.all(np.abs(wts[:, :4] - 0.25) <= 1e-15) and np.all(wts[:, 4:] == 0.0)
    finally:
        bg.moe_plan_destroy(plan)


@pytest.mark.parametrize("T,path", [(128, 1), (4, 2), (4, 1)])
def test_operand_range_is_flagged(T, path):
    """Inputs outside the fp16 operand contract of the expert GEMMs latch an
    error that moe_get_error reports as MOE_ERR_OPERAND_RANGE (6): a token
    value above 65504 (checked on every call), and a weight set with a scale
    below 2^-14 (checked the first time a plan sees the set). In-contract
    inputs report 0, as in every other test of this suite."""
    w = dataclasses.replace(WL["t128_uniform"], tokens=T)
    c = Case(w, gap=False)
    plan = make_plan(w, path)
    try:
        run_layer(c, plan)                                  # in contract: status 0
        x_big = c.x.clone()
        x_big[T // 2, 17] = 70000.0                         # bf16 70144: saturates in fp16
        y = torch.empty(c.x.shape, dtype=torch.float32, device="cuda")
        bg.moe_forward_layer(plan, x_big, T, c.L.router_w, c.L.router_bias, c.L.routed_c,
                             c.L.shared_c, y)
        assert bg.moe_get_error(plan) == 6
        run_layer(c, plan)                                  # cleared; x back in range
        # a subnormal-in-fp16 scale in a fresh copy of the up matrix's scales
        up_s = c.L.routed["up"][1].clone()
        up_s[3, 5, 2] = 1e-6
        routed = bg.experts(c.L.routed["gate"], (c.L.routed["up"][0], up_s, c.L.routed["up"][2]),
                            c.L.routed["down"])
        bg.moe_forward_layer(plan, c.x, T, c.L.router_w, c.L.router_bias, routed, c.L.shared_c, y)
        torch.cuda.synchronize()
        assert bg.moe_get_error(plan) == 6
        # a bias of magnitude 2^11 in the shared expert's down matrix
        sd_b = c.L.shared["down"][2].clone()
        sd_b[0, 100, 3] = 2048.0
        shared = bg.experts(c.L.shared["gate"], c.L.shared["up"],
                            (c.L.shared["down"][0], c.L.shared["down"][1], sd_b))
        bg.moe_forward_layer(plan, c.x, T, c.L.router_w, c.L.router_bias, c.L.routed_c, shared, y)
        assert bg.moe_get_error(plan) == 6
        assert bg.moe_get_error(plan) == 0
    finally:
        bg.moe_plan_destroy(plan)


@pytest.mark.parametrize("T", [4, 512])
def test_no_host_sync_inside_a_layer(T):
    """A layer call returns while the device is still busy: the stream is
    held by a kernel that spins for about a second (torch.cuda._sleep), the
    layer is enqueued behind it, and the stream must still report work
    pending when the call has returned (a host sync inside the call would
    have waited for the sleep). Warm calls first, so that one-time work
    (module loading, tensor maps, the weight range check) is done."""
    w = dataclasses.replace(WL["t512_zipf"], tokens=T)
    c = Case(w, gap=False)
    plan = make_plan(w)
    try:
        y = torch.empty(c.x.shape, dtype=torch.float32, device="cuda")
        xs, xn = c.x.clone(), torch.empty_like(c.x)
        layers = bg.moe_layers([c.L])
        for _ in range(2):
            bg.moe_forward_layer(plan, c.x, T, c.L.router_w, c.L.router_bias, c.L.routed_c,
                                 c.L.shared_c, y)
            bg.moe_forward_stack(plan, xs, xn, T, layers, 0.1)
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        for call in ("layer", "stack"):
            torch.cuda._sleep(2_000_000_000)              # ~1 s of device time
            if call == "layer":
                bg.moe_forward_layer(plan, c.x, T, c.L.router_w, c.L.router_bias, c.L.routed_c,
                                     c.L.shared_c, y)
            else:
                bg.moe_forward_stack(plan, xs, xn, T, layers, 0.1)
            assert not stream.query(), f"{call}: the call waited for the device"
            torch.cuda.synchronize()
        assert bg.moe_get_error(plan) == 0
    finally:
        bg.moe_plan_destroy(plan)


@pytest.mark.parametrize("T", [1, 4, 8])
@pytest.mark.parametrize("path", [0, 1])
def test_decode_sized_layer(T, path):
    w = dataclasses.replace(WL["decode_t8_l40"], tokens=T, layers=1)
    c = Case(w)
    plan = make_plan(w, path)
    try:
        y = run_layer(c, plan)
        assert bg.moe_last_gemm_path(plan) == (path if path else 2)
        parity.check_y(y.double().cpu().numpy(), c.oracle_layer()["y"])
    finally:
        bg.moe_plan_destroy(plan)


@pytest.mark.parametrize("T,shared,path,routing", [
    (37, True, 1, "zipf"), (37, True, 2, "zipf"), (300, False, 1, "uniform"),
    (300, False, 2, "uniform"), (129, True, 0, "zipf"), (300, False, 3, "uniform"),
    (600, True, 1, "zipf"),
])
def test_small_shapes_ragged(T, shared, path, routing):
    sh = dataclasses.replace(SMALL, has_shared=shared)
    w = synth.Workload(f"small{T}", T, 1, routing, seed=77 + T, shape=sh)
    c = Case(w)
    plan = make_plan(w, path)
    try:
        r = bg.moe_route(plan, c.x, T, c.L.router_w, c.L.router_bias)
        g = parity.routing_to_numpy(r, T, sh.top_k, sh.num_experts)
        _, idx, _, _, maps = c.oracle_route()
        assert np.array_equal(g["topk_idx"], idx)
        assert np.array_equal(g["perm"], maps["perm"])
        assert np.array_equal(g["block_map"], maps["block_map"])
        y = run_layer(c, plan)
        parity.check_y(y.double().cpu().numpy(), c.oracle_layer()["y"])
    finally:
        bg.moe_plan_destroy(plan)


def test_ffn_on_caller_routing():
    # moe_grouped_w4_ffn on a routing the caller supplies (the oracle's)
    w = WL["t128_uniform"]
    c = Case(w)
    sh = w.shape
    _, idx, wts, _, maps = c.oracle_route()
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    bufs = dict(topk_idx=dev(idx.astype(np.int32)), topk_w=dev(wts.astype(np.float32)),
                counts=dev(maps["counts"]), offsets=dev(maps["offsets"]),
                tile_offsets=dev(maps["tile_offsets"]), perm=dev(maps["perm"]),
                inv=dev(maps["inv"]), block_map=dev(maps["block_map"].reshape(-1)),
                num_tiles=dev(np.array([maps["num_tiles"]], np.int32)))
    r = bg.MoeRouting(**{k: v.data_ptr() for k, v in bufs.items()}, logits=None)
    plan = make_plan(w)
    try:
        y = torch.empty(c.x.shape, dtype=torch.float32, device="cuda")
        bg.moe_grouped_w4_ffn(plan, c.x, w.tokens, r, c.L.routed_c, c.L.shared_c, y)
        torch.cuda.synchronize()
        parity.check_y(y.double().cpu().numpy(), c.oracle_layer()["y"])
    finally:
        bg.moe_plan_destroy(plan)


@pytest.mark.parametrize("name", ["t512_zipf", "t2048_uniform"])
def test_routing_fused_gather_matches_gather_launch(name):
    # moe_forward_layer lets the cooperative routing launch write the gathered
    # rows; moe_route + moe_grouped_w4_ffn runs the separate gather kernel.
    w = WL[name]
    c = Case(w, gap=False)
    plan = make_plan(w)
    try:
        y1 = run_layer(c, plan).cpu().numpy()
        r = bg.moe_route(plan, c.x, w.tokens, c.L.router_w, c.L.router_bias)
        y2 = torch.empty(c.x.shape, dtype=torch.float32, device="cuda")
        bg.moe_grouped_w4_ffn(plan, c.x, w.tokens, r, c.L.routed_c, c.L.shared_c, y2)
        torch.cuda.synchronize()
        assert bg.moe_get_error(plan) == 0
        assert np.array_equal(y1, y2.cpu().numpy())
    finally:
        bg.moe_plan_destroy(plan)


@pytest.mark.parametrize("path", [1, 2, 3])
def test_deterministic(path):
    w = WL["t512_zipf"]
    c = Case(w, gap=False)
    plan = make_plan(w, path)
    try:
        y1 = run_layer(c, plan).clone()
        a1 = y1.cpu().numpy()
        y2 = run_layer(c, plan)
        assert np.array_equal(a1, y2.cpu().numpy())
    finally:
        bg.moe_plan_destroy(plan)


def test_device_timeout_is_reported_and_context_survives():
    w = WL["t128_uniform"]
    plan = make_plan(w)
    try:
        assert bg.moe_get_error(plan) == 0
        bg.moe_debug_wait_timeout(plan, 20000)          # 20 ms limit, never satisfied
        assert bg.moe_get_error(plan) == 5              # MOE_ERR_DEVICE_TIMEOUT
        assert bg.moe_get_error(plan) == 0              # cleared
        c = Case(w, gap=False)
        run_layer(c, plan)                              # context still usable
    finally:
        bg.moe_plan_destroy(plan)


def test_host_argument_errors():
    w = WL["t128_uniform"]
    plan = make_plan(w)
    try:
        c = Case(w, gap=False)
        y = torch.empty(c.x.shape, dtype=torch.float32, device="cuda")
        with pytest.raises(bg.MoeError) as ei:
            bg.moe_forward_layer(plan, c.x, w.tokens + 1, c.L.router_w, None, c.L.routed_c,
                                 c.L.shared_c, y)
        assert ei.value.status == 4                      # capacity
        with pytest.raises(bg.MoeError) as ei:
            bg.moe_forward_layer(plan, c.x, 0, c.L.router_w, None, c.L.routed_c, c.L.shared_c, y)
        assert ei.value.status == 1
        with pytest.raises(bg.MoeError) as ei:              # y aliases x
            bg.moe_forward_layer(plan, c.x, 8, c.L.router_w, None, c.L.routed_c, c.L.shared_c,
                                 c.x)
        assert ei.value.status == 1
        with pytest.raises(bg.MoeError) as ei:              # misaligned x
            bg.moe_forward_layer(plan, c.x.view(-1)[1:].data_ptr(), 8, c.L.router_w, None,
                                 c.L.routed_c, c.L.shared_c, y)
        assert ei.value.status == 1
        with pytest.raises(bg.MoeError) as ei:              # shared set given but plan has none
            bg.moe_forward_layer(plan, c.x, 8, c.L.router_w, None, c.L.routed_c, None, y)
        assert ei.value.status == 1
    finally:
        bg.moe_plan_destroy(plan)
