"""moe_route_noalloc (routing with no device allocation inside the library)
against moe_route, through the C ABI.

Callers that cannot call cudaMalloc -- code inside another framework's
memory pool, allocator-less runtimes -- pass every output
buffer themselves; the library's only scratch for this call is a fixed
device array. The test allocates the output buffers (the entry point does
not), runs two calls in a row with different inputs, and requires the same
routing as the plan-based entry point: integer arrays exactly, top-k weights
within the 1e-5 tolerance of the other routing tests.
"""
import numpy as np
import pytest
import torch

from bit_grouped_gemm_gb300 import binding as bg
from bit_grouped_gemm_gb300 import stack, synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bit_grouped_gemm_gb300 import build
    build.build()
    bg.load_library()


def caller_buffers(T, k, E):
    return parity.caller_routing_buffers(T, k, E)


@pytest.mark.parametrize("name", ["t512_zipf", "t128_uniform"])
def test_noalloc_routing_matches_moe_route_twice(name):
    w = synth.standard_workloads()[name]
    sh = w.shape
    layers = [stack.make_layer(w, 0, "cuda"), stack.make_layer(w, 1, "cuda")]
    xs = [synth.tokens_x(w, "cuda"), synth.decode_pool(w, 1, "cuda")[0]]
    plan = bg.moe_plan_create(bg.plan_desc(max_tokens=w.tokens), 0)
    try:
        for call in range(2):                          # two calls in a row
            L, x = layers[call], xs[call]
            ref = parity.routing_to_numpy(
                bg.moe_route(plan, x, w.tokens, L.router_w, L.router_bias),
                w.tokens, sh.top_k, sh.num_experts)
            bufs, r = caller_buffers(w.tokens, sh.top_k, sh.num_experts)
            bg.moe_route_noalloc(x, w.tokens, sh.hidden, L.router_w, L.router_bias,
                                 sh.num_experts, sh.top_k, r)
            got = parity.routing_to_numpy(r, w.tokens, sh.top_k, sh.num_experts)
            for key in ("topk_idx", "counts", "offsets", "tile_offsets", "perm", "inv",
                        "block_map"):
                assert np.array_equal(got[key], ref[key]), (call, key)
            assert got["num_tiles"] == ref["num_tiles"]
            assert np.abs(got["topk_w"] - ref["topk_w"]).max() <= parity.W_TOL
            assert np.abs(got["logits"] - ref["logits"]).max() <= 1e-6
    finally:
        bg.moe_plan_destroy(plan)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    w = synth.standard_workloads()["t128_uniform"]
    L = stack.make_layer(w, 0, "cuda")
    x = torch.zeros(4097, 2048, dtype=torch.bfloat16, device="cuda")
    _, r = caller_buffers(16, 8, 256)
    with pytest.raises(bg.MoeError) as ei:
        bg.moe_route_noalloc(x, 4097, 2048, L.router_w, None, 256, 8, r)
    assert ei.value.status == 4                        # MOE_ERR_CAPACITY


# A plan routes a batch of at most 16 tokens in one launch (logits GEMV, then
# top-k, scans, block map and scatter by the CTA that finishes last), and a
# larger batch in two (the logits GEMM, then one cooperative launch for
# selection through scatter); moe_route_noalloc always takes the separate
# launches. Same arithmetic in the same order: every array, logits and
# weights included, must agree bit for bit, over each width the fused
# kernels are specialised on, with and without a bias, on two calls in a row
# (the arrival counter and the generation word rearm).
FUSED_CASES = [
    # T, hidden, experts, top_k, routing
    (1, 2048, 256, 8, "zipf"), (5, 2048, 256, 8, "uniform"), (16, 2048, 256, 8, "zipf"),
    (3, 1024, 512, 8, "uniform"), (16, 512, 8, 2, "zipf"), (9, 1024, 64, 32, "uniform"),
    (17, 2048, 256, 8, "zipf"), (300, 1024, 512, 8, "zipf"), (2048, 2048, 256, 8, "uniform"),
    (4096, 2048, 256, 8, "zipf"), (999, 512, 8, 2, "uniform"), (77, 512, 64, 32, "zipf"),
]


@pytest.mark.parametrize("T,H,E,k,routing", FUSED_CASES)
def test_fused_routing_matches_separate_launches(T, H, E, k, routing):
    sh = synth.MoEShape(hidden=H, inter=256, num_experts=E, top_k=k)
    w = synth.Workload(f"fused{T}", T, 2, routing, seed=500 + T + E, shape=sh)
    plan = bg.moe_plan_create(bg.plan_desc(hidden=H, inter=256, num_experts=E, top_k=k,
                                           max_tokens=T), 0)
    try:
        for call in range(2):
            wr = synth.router_weight(w, call, "cuda")
            rb = synth.router_bias(w, call, "cuda")
            x = synth.decode_pool(w, 2, "cuda")[call]
            ref = parity.routing_to_numpy(bg.moe_route(plan, x, T, wr, rb), T, k, E)
            bufs, r = caller_buffers(T, k, E)
            bg.moe_route_noalloc(x, T, H, wr, rb, E, k, r)
            got = parity.routing_to_numpy(r, T, k, E)
            for key in ("logits", "topk_idx", "topk_w", "counts", "offsets", "tile_offsets",
                        "perm", "inv", "block_map"):
                assert np.array_equal(got[key], ref[key]), (call, key)
            assert got["num_tiles"] == ref["num_tiles"]
    finally:
        bg.moe_plan_destroy(plan)


def test_noalloc_device_timeout_is_reported_and_cleared():
    """The allocation-free routing has its own device error word (it has no
    plan): a bounded wait that runs out is reported by
    moe_route_noalloc_get_error, which also clears it, and routing still
    works afterwards. The wait is made to run out by a kernel whose barrier
    nothing signals (20 ms limit): no fault, no hang."""
    assert bg.moe_route_noalloc_get_error() == 0
    bg.moe_route_noalloc_debug_wait_timeout(20000)
    assert bg.moe_route_noalloc_get_error() == 5           # MOE_ERR_DEVICE_TIMEOUT
    assert bg.moe_route_noalloc_get_error() == 0           # cleared
    w = synth.standard_workloads()["t128_uniform"]
    sh = w.shape
    L = stack.make_layer(w, 0, "cuda")
    x = synth.tokens_x(w, "cuda")
    _, r = caller_buffers(w.tokens, sh.top_k, sh.num_experts)
    bg.moe_route_noalloc(x, w.tokens, sh.hidden, L.router_w, L.router_bias, sh.num_experts,
                         sh.top_k, r)
    got = parity.routing_to_numpy(r, w.tokens, sh.top_k, sh.num_experts)
    assert got["offsets"][-1] == w.tokens * sh.top_k
    assert bg.moe_route_noalloc_get_error() == 0
