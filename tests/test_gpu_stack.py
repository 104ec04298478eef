"""GPU parity of the stacked layers:
    xn = rmsnorm(x); y = moe(xn); x <- bf16(x + y/sqrt(L)); xn <- rmsnorm(x)

The GPU chain runs through exactly the calls the benchmark times (for
prefill moe_forward_layer_residual per layer, the combine fused with the
stack update, as moe_forward_stack issues it; for decode the same calls the
replayed CUDA graph holds). The oracle follows a set of token rows through
all layers on its own, in fp64, from the generator's inputs; no oracle input
ever comes from the GPU. At each layer the GPU also runs the layer, with the
same call, on a copy of its batch in which the followed rows are replaced by
the oracle's rows (same T, same grid; the rest of the batch keeps the GPU's
routing context). On those rows:
  * routing indices must equal the oracle's wherever the oracle's 8th/9th
    logit gap is >= 1e-3;
  * the layer output y (rebuilt from the plan's scratch exactly as the fused
    combine adds it) must satisfy max|y_gpu - y_oracle| <= 2e-2 *
    rms(y_oracle) over the compared rows of the layer;
  * the updated residual row must be y's update, bf16(x + y/sqrt(L)), to
    within half a bf16 unit in the last place (plus the FP32 rounding before
    it), and the next layer's input its RMS norm to within one unit.
The GPU's own chain is checked at every layer for the invariants any correct
routing map has.

Rows followed at T = 4096: for layer 0 (whose routing the oracle computes on
all rows beforehand), the last token of every active expert (so every
expert's last, partial tile holds a compared row) and the first token of
every tile of the most loaded expert; every 16th token (so every tile of a
hot expert holds several, at every layer); and the last 32 tokens. Decode
batches (T = 1, 4, 8) follow every row.
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
        sel = torch.tensor(need, dtype=torch.int64, device=q.device)
        qh[need] = parity.words(q[sel])
        shh[need] = parity.bits(s[sel])
        bh[need] = parity.bits(b[sel])
        routed[m] = (qh, shh, bh)
    shared = parity.host_set(L.shared) if L.shared is not None else None
    return orc.moe_rows(xn_bits, wr, rb, routed, shared, sh.top_k, sh.group_size,
                        nthreads=NTHREADS)


def to_dev_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(b.view(np.int16).copy()).cuda().view(torch.bfloat16)


def bits_f64(b: np.ndarray) -> np.ndarray:
    return parity.bf16_f64(b)


def tile_coverage(g: dict, rows_ok: np.ndarray, k: int):
    """From a routing result: (last tiles of active experts holding a compared
    row, active experts, tiles of the most loaded expert holding a compared
    row, its tiles)."""
    bmap, inv, cnt = g["block_map"], g["inv"], g["counts"]
    pos = inv.reshape(-1, k)[rows_ok].reshape(-1)
    starts = bmap[:, 1]
    tile_of = np.searchsorted(starts, pos, side="right") - 1
    covered = np.zeros(len(bmap), bool)
    covered[tile_of] = True
    last = {}
    for t, (e, _, _) in enumerate(bmap):
        last[int(e)] = t
    n_last = sum(covered[t] for t in last.values())
    hot = int(np.argmax(cnt))
    hot_tiles = [t for t, (e, _, _) in enumerate(bmap) if e == hot]
    return int(n_last), len(last), int(covered[hot_tiles].sum()), len(hot_tiles)


def prefill_rows(w: synth.Workload, L0: stack.DeviceLayer) -> np.ndarray:
    """The token rows the 40-layer prefill chain follows (module docstring)."""
    orc = oracle.get()
    sh = w.shape
    T, k = w.tokens, sh.top_k
    xn0 = orc.rmsnorm(parity.bits(synth.tokens_x(w, "cpu")))
    rb = None if L0.router_bias is None else L0.router_bias.cpu().numpy()
    idx, _, gap = orc.topk(parity.router_logits_mt(orc, xn0, parity.bits(L0.router_w), rb), k)
    maps = orc.route_maps(idx, sh.num_experts, 128)
    off, perm, cnt = maps["offsets"], maps["perm"], maps["counts"]
    rows = set(range(0, T, 16)) | set(range(T - 32, T))
    for e in np.nonzero(cnt)[0]:
        # the last token of the expert's last tile whose gap allows comparison
        first_last_tile = off[e] + 128 * ((cnt[e] - 1) // 128)
        for p in range(off[e + 1] - 1, first_last_tile - 1, -1):
            t = perm[p] // k
            if gap[t] >= parity.GAP_MIN:
                rows.add(int(t))
                break
    hot = int(np.argmax(cnt))
    for p in range(off[hot], off[hot + 1], 128):
        rows.add(int(perm[p] // k))
    return np.array(sorted(rows), np.int32)


def run_chain_check(w: synth.Workload, rows: np.ndarray, layers=None):
    """The chain check of the module docstring; returns per-layer stats
    (layer, compared rows, y ratio, last tiles covered, active experts, hot
    tiles covered, hot tiles)."""
    sh = w.shape
    T, k, H = w.tokens, sh.top_k, sh.hidden
    layers = layers if layers is not None else stack.make_layers(w, "cuda")
    plan = bg.moe_plan_create(bg.plan_desc(sh.hidden, sh.inter, sh.num_experts, sh.top_k,
                                           sh.group_size, int(sh.has_shared), T), 0)
    alpha = stack.residual_alpha(w.layers)
    orc = oracle.get()
    stats = []
    try:
        x = synth.tokens_x(w, "cuda")
        xn = torch.empty_like(x)
        xo = parity.bits(x)[rows]                    # the oracle's own chain
        bg.moe_residual_add(plan, x, None, T, 0.0, x, xn)
        rows_t = torch.from_numpy(rows.astype(np.int64)).cuda()
        for li, L in enumerate(layers):
            # the GPU chain's routing invariants
            r = bg.moe_route(plan, xn, T, L.router_w, L.router_bias)
            g = parity.routing_to_numpy(r, T, k, sh.num_experts)
            check_route_invariants(g, g["topk_idx"], sh.num_experts, 128)
            # the layer on the oracle's rows, through the timed call
            xon = orc.rmsnorm(xo)
            xin = xn.clone()
            xin[rows_t] = to_dev_bits(xon)
            x_chk = x.clone()
            x_chk[rows_t] = to_dev_bits(xo)
            xn_chk = torch.empty_like(x)
            rc = bg.moe_route(plan, xin, T, L.router_w, L.router_bias)   # the routing pointers
            bg.moe_forward_layer_residual(plan, xin, T, L.router_w, L.router_bias, L.routed_c,
                                          L.shared_c, alpha, x_chk, xn_chk)
            gc = parity.routing_to_numpy(rc, T, k, sh.num_experts)
            y_gpu = parity.layer_output_from_scratch(plan, gc["inv"], rows, T, k, H,
                                                     sh.has_shared)
            o = oracle_layer_for_rows(L, xon, sh)
            ok = o["gap"] >= parity.GAP_MIN
            assert np.array_equal(gc["topk_idx"][rows][ok], o["topk_idx"][ok]), li
            # (a layer where no followed row has the gap compares no output;
            # the chains still advance, each with its own routing)
            ratio = parity.check_y(y_gpu[ok].astype(np.float64), o["y"][ok]) if ok.any() else 0.0
            # the fused stack update on the same rows
            xc = bits_f64(parity.bits(x_chk)[rows])
            want = bits_f64(xo) + np.float64(np.float32(alpha)) * y_gpu.astype(np.float64)
            slack = 0.5 * parity.bf16_ulp(np.maximum(np.abs(xc), np.abs(want))) * (1 + 2.0 ** -15)
            assert np.all(np.abs(xc - want) <= slack + 1e-30), li
            xn_want = bits_f64(orc.rmsnorm(parity.bits(x_chk)[rows]))
            xn_got = bits_f64(parity.bits(xn_chk)[rows])
            assert np.all(np.abs(xn_got - xn_want) <= parity.bf16_ulp(xn_want) + 1e-30), li
            cov = tile_coverage(gc, rows[ok], k) if ok.any() else (0, 0, 0, 0)
            stats.append((li, int(ok.sum()), ratio) + cov)
            # advance both chains: the GPU by the timed call, the oracle by its own update
            bg.moe_forward_layer_residual(plan, xn, T, L.router_w, L.router_bias, L.routed_c,
                                          L.shared_c, alpha, x, xn)
            xo = orc.residual(xo, o["y"], alpha)
        assert bg.moe_get_error(plan) == 0
        assert np.isfinite(x.float().cpu().numpy()).all()
        return stats
    finally:
        bg.moe_plan_destroy(plan)


def test_prefill_stack_t4096_l40_chain():
    w = synth.standard_workloads()["prefill_t4096_l40_zipf"]
    layers = stack.make_layers(w, "cuda")
    rows = prefill_rows(w, layers[0])
    assert len(rows) >= 256
    stats = run_chain_check(w, rows, layers)
    print("layer, compared rows, y ratio, last tiles covered/active, hot tiles covered/all")
    for st in stats:
        print(f"  {st[0]:2d} {st[1]:4d} {st[2]:.2e} {st[3]}/{st[4]} {st[5]}/{st[6]}")
    assert sum(st[1] for st in stats) >= 0.9 * len(rows) * w.layers, stats
    # layer 0: every active expert's last tile holds a compared row
    assert stats[0][3] >= stats[0][4] - 2, stats[0]
    # every layer: every tile of the most loaded expert holds a compared row
    assert all(st[5] == st[6] for st in stats), stats


@pytest.mark.parametrize("T", [1, 4, 8])
def test_decode_stack_l40_chain(T):
    w = synth.standard_workloads()[f"decode_t{T}_l40"]
    stats = run_chain_check(w, np.arange(T, dtype=np.int32))
    assert sum(st[1] for st in stats) >= 0.9 * T * w.layers, stats


def routing_pointers(plan, x, T, L):
    """Device addresses of the plan's routing arrays (stable for a plan)."""
    return bg.moe_route(plan, x, T, L.router_w, L.router_bias)


def fused_layer_chain(w, layers, alpha):
    """The fused decode layer (moe_forward_stack on a chunk of at most 8
    tokens: router, top-k, gate/up, down, combine and stack update in one
    launch per layer) against the oracle over `layers` of the 40-layer stack
    (alpha the stack's residual scale). At every
    layer the GPU runs that one layer on the oracle's residual rows; its
    routing must equal the oracle's (rows with the gap), its FP32 block output
    (kept in the plan's scratch) must be within 2e-2 * rms of the oracle's,
    and the updated rows must be bf16(x + y/sqrt(L)) of that output."""
    sh = w.shape
    T, k, H = w.tokens, sh.top_k, sh.hidden
    plan = bg.moe_plan_create(bg.plan_desc(sh.hidden, sh.inter, sh.num_experts, sh.top_k,
                                           sh.group_size, int(sh.has_shared), T), 0)
    orc = oracle.get()
    try:
        x = synth.decode_pool(w, 1, "cuda")[0].contiguous()
        xn = torch.empty_like(x)
        r = routing_pointers(plan, x, T, layers[0])
        y_view = parity.device_view(bg.moe_debug_buffer(plan, 3), T * H, torch.float32)
        xo = parity.bits(x)
        compared = 0
        for li, L in enumerate(layers):
            one = bg.moe_layers([L])
            x_chk = to_dev_bits(xo)
            bg.moe_forward_stack(plan, x_chk, xn, T, one, alpha)
            torch.cuda.synchronize()
            assert bg.moe_last_gemm_path(plan) == 3
            gidx = parity.device_view(r.topk_idx, T * k, torch.int32).cpu().numpy().reshape(T, k)
            y_gpu = y_view.cpu().numpy().reshape(T, H)
            o = oracle_layer_for_rows(L, orc.rmsnorm(xo), sh)
            ok = o["gap"] >= parity.GAP_MIN
            assert np.array_equal(gidx[ok], o["topk_idx"][ok]), li
            if ok.any():
                parity.check_y(y_gpu[ok].astype(np.float64), o["y"][ok])
            compared += int(ok.sum())
            xc = bits_f64(parity.bits(x_chk))
            want = bits_f64(xo) + np.float64(np.float32(alpha)) * y_gpu.astype(np.float64)
            slack = 0.5 * parity.bf16_ulp(np.maximum(np.abs(xc), np.abs(want))) * (1 + 2.0 ** -15)
            assert np.all(np.abs(xc - want) <= slack + 1e-30), li
            assert np.array_equal(parity.bits(xn), orc.rmsnorm(parity.bits(x_chk))) or np.all(
                np.abs(bits_f64(parity.bits(xn)) - bits_f64(orc.rmsnorm(parity.bits(x_chk))))
                <= parity.bf16_ulp(bits_f64(orc.rmsnorm(parity.bits(x_chk)))) + 1e-30), li
            xo = orc.residual(xo, o["y"], alpha)
        assert compared >= 0.9 * T * len(layers)
        assert bg.moe_get_error(plan) == 0
    finally:
        bg.moe_plan_destroy(plan)


@pytest.mark.parametrize("T", [1, 4, 8])
def test_decode_fused_layer_chain(T):
    """The chain above over the whole 40-layer stack at the benchmark's batch
    sizes."""
    w = synth.standard_workloads()[f"decode_t{T}_l40"]
    fused_layer_chain(w, stack.make_layers(w, "cuda"), stack.residual_alpha(w.layers))


@pytest.mark.parametrize("T", [2, 3, 5, 7])
def test_decode_fused_layer_chain_other_sizes(T):
    """The same chain over the first 6 layers of the stack at batch sizes the
    benchmark skips: 2, and odd token counts, where a slot's last pair of
    MMA columns holds one token."""
    w = dataclasses.replace(synth.standard_workloads()["decode_t8_l40"], name=f"decode_t{T}_l40",
                            tokens=T)
    fused_layer_chain(w, [stack.make_layer(w, li, "cuda") for li in range(6)],
                      stack.residual_alpha(w.layers))


def test_decode_fused_after_timeout_reset():
    """A bounded wait that runs out latches MOE_ERR_DEVICE_TIMEOUT; clearing it
    also resets the fused decode layer's launch count and its launch-tagged
    router logits, so the fused steps that follow give the bits they gave
    before the error (and no stale logits are taken for new ones)."""
    w = synth.standard_workloads()["decode_t4_l40"]
    sh = w.shape
    layers = [stack.make_layer(w, li, "cuda") for li in range(3)]
    plan = bg.moe_plan_create(bg.plan_desc(sh.hidden, sh.inter, sh.num_experts, sh.top_k,
                                           sh.group_size, int(sh.has_shared), w.tokens), 0)
    alpha = stack.residual_alpha(w.layers)
    try:
        x0 = synth.decode_pool(w, 1, "cuda")[0].contiguous()
        xn = torch.empty_like(x0)
        arr = bg.moe_layers(layers)

        def two_steps():
            x = x0.clone()
            bg.moe_forward_stack(plan, x, xn, w.tokens, arr, alpha)
            bg.moe_forward_stack(plan, x, xn, w.tokens, arr, alpha)
            torch.cuda.synchronize()
            return x.view(torch.int16).cpu().numpy()

        a = two_steps()
        assert bg.moe_last_gemm_path(plan) == 3
        assert bg.moe_get_error(plan) == 0
        bg.moe_debug_wait_timeout(plan, 20000)      # 20 ms limit, never satisfied
        assert bg.moe_get_error(plan) == 5          # MOE_ERR_DEVICE_TIMEOUT, cleared
        b = two_steps()
        assert bg.moe_get_error(plan) == 0
        assert np.array_equal(a, b)
    finally:
        bg.moe_plan_destroy(plan)


@pytest.mark.parametrize("T", [1, 8])
def test_decode_fused_stack_matches_layer_by_layer(T):
    """One moe_forward_stack call over the 40 layers (the launch sequence the
    decode benchmark replays) gives the bits of 40 one-layer calls, which the
    chain test above compares with the oracle layer by layer."""
    w = synth.standard_workloads()[f"decode_t{T}_l40"]
    sh = w.shape
    layers = stack.make_layers(w, "cuda")
    plan = bg.moe_plan_create(bg.plan_desc(sh.hidden, sh.inter, sh.num_experts, sh.top_k,
                                           sh.group_size, int(sh.has_shared), T), 0)
    alpha = stack.residual_alpha(w.layers)
    try:
        x0 = synth.decode_pool(w, 1, "cuda")[0].contiguous()
        xn = torch.empty_like(x0)
        a = x0.clone()
        bg.moe_forward_stack(plan, a, xn, T, bg.moe_layers(layers), alpha)
        b = x0.clone()
        for L in layers:
            bg.moe_forward_stack(plan, b, xn, T, bg.moe_layers([L]), alpha)
        torch.cuda.synchronize()
        assert np.array_equal(a.view(torch.int16).cpu().numpy(), b.view(torch.int16).cpu().numpy())
        assert bg.moe_get_error(plan) == 0
    finally:
        bg.moe_plan_destroy(plan)


@pytest.mark.parametrize("T,fused", [(1, True), (8, True), (8, False), (16, True)])
def test_decode_graph_replay_matches_eager(T, fused):
    """The decode benchmark replays the whole 40-layer step from one CUDA
    graph; the replay gives the bits of the same calls issued eagerly (which
    the chain tests above compare with the oracle): moe_forward_stack (the
    fused decode layer at T <= 8, the general small-M path at T = 16), or the
    per-layer calls."""
    w = dataclasses.replace(synth.standard_workloads()["decode_t8_l40"], tokens=T)
    sh = w.shape
    layers = stack.make_layers(w, "cuda")
    plan = bg.moe_plan_create(bg.plan_desc(sh.hidden, sh.inter, sh.num_experts, sh.top_k,
                                           sh.group_size, int(sh.has_shared), T), 0)
    try:
        pool = synth.decode_pool(w, 4, "cuda")
        alpha = stack.residual_alpha(w.layers)
        x = torch.empty((T, sh.hidden), dtype=torch.bfloat16, device="cuda")
        xn = torch.empty_like(x)
        y = torch.empty(x.shape, dtype=torch.float32, device="cuda")
        arr = bg.moe_layers(layers)

        def step():
            if fused:
                bg.moe_forward_stack(plan, x, xn, T, arr, alpha)
            else:
                stack.run_stack(plan, x, xn, layers, T, y, alpha)

        x.copy_(pool[0])
        step()                                                 # warm (one-time work)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="thread_local"):
            step()
        for i in (1, 2, 3):
            x.copy_(pool[i])
            step()
            torch.cuda.synchronize()
            eager = x.view(torch.int16).cpu().numpy().copy()
            x.copy_(pool[i])
            graph.replay()
            torch.cuda.synchronize()
            assert np.array_equal(x.view(torch.int16).cpu().numpy(), eager), i
        assert bg.moe_get_error(plan) == 0
    finally:
        bg.moe_plan_destroy(plan)


@pytest.mark.parametrize("chunk", [256])
def test_chunked_prefill_parity(chunk):
    """moe_forward_stack on a prompt longer than the plan's capacity (600
    tokens in chunks of 256, 256 and a ragged 88) against the oracle, layer by
    layer over 3 layers: at each layer the GPU runs moe_forward_stack for that
    one layer on its batch with the followed rows replaced by the oracle's
    residual rows (rows in every chunk, and every row of the last one), and
    the updated rows must satisfy |x_gpu - x_oracle| <= sqrt(1/L) * 2e-2 *
    rms(y_oracle) + one bf16 unit (both sides round x + y/sqrt(L) once to
    bf16 after outputs within the layer tolerance)."""
    T = 600
    w = dataclasses.replace(synth.standard_workloads()["prefill_t4096_l40_zipf"], tokens=T,
                            layers=3)
    sh = w.shape
    layers = stack.make_layers(w, "cuda")
    alpha = stack.residual_alpha(40)
    rows = np.array(sorted({0, 1, 100, 255, 256, 300, 511} | set(range(512, T))), np.int32)
    rows_t = torch.from_numpy(rows.astype(np.int64)).cuda()
    plan = bg.moe_plan_create(bg.plan_desc(sh.hidden, sh.inter, sh.num_experts, sh.top_k,
                                           sh.group_size, int(sh.has_shared), chunk), 0)
    orc = oracle.get()
    try:
        x = synth.tokens_x(w, "cuda")
        xn = torch.empty((chunk, sh.hidden), dtype=x.dtype, device="cuda")
        xo = parity.bits(x)[rows]
        for li, L in enumerate(layers):
            one = bg.moe_layers([L])
            x_chk = x.clone()
            x_chk[rows_t] = to_dev_bits(xo)
            bg.moe_forward_stack(plan, x_chk, xn, T, one, alpha)
            o = oracle_layer_for_rows(L, orc.rmsnorm(xo), sh)
            xo_next = orc.residual(xo, o["y"], alpha)
            ok = o["gap"] >= parity.GAP_MIN
            got = bits_f64(parity.bits(x_chk)[rows])[ok]
            want = bits_f64(xo_next)[ok]
            rms = float(np.sqrt(np.mean(o["y"][ok] ** 2)))
            bound = alpha * parity.Y_TOL * rms + parity.bf16_ulp(np.maximum(np.abs(got),
                                                                            np.abs(want)))
            assert np.all(np.abs(got - want) <= bound), li
            assert ok.sum() >= 0.9 * len(rows)
            bg.moe_forward_stack(plan, x, xn, T, one, alpha)        # the GPU's own chain
            xo = xo_next
        assert bg.moe_get_error(plan) == 0
    finally:
        bg.moe_plan_destroy(plan)


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
    tensor-core path like the whole prompt. The split of the last round of
    units is off in both plans (it sums a tile's K range in pieces, so a
    token's last bits depend on where its tile falls in the deal)."""
    T = 600
    w = dataclasses.replace(synth.standard_workloads()["prefill_t4096_l40_zipf"], tokens=T, layers=3)
    sh = w.shape
    layers = stack.make_layers(w, "cuda")
    mk = lambda m: bg.moe_plan_create(bg.plan_desc(sh.hidden, sh.inter, sh.num_experts, sh.top_k,
                                                   sh.group_size, int(sh.has_shared), m), 0)
    whole, chunked = mk(T), mk(chunk)
    try:
        bg.moe_set_tail_split(whole, False)
        bg.moe_set_tail_split(chunked, False)
        x0 = synth.tokens_x(w, "cuda")
        a = _stack_bits(whole, w, layers, T, True, x0)
        b = _stack_bits(chunked, w, layers, T, True, x0)
        assert np.array_equal(a, b)
    finally:
        bg.moe_plan_destroy(whole)
        bg.moe_plan_destroy(chunked)
