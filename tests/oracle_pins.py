"""Pins of the fp64 oracle to facts other than itself.

Each ``pin_*`` function takes a loaded ``oracle.Oracle`` and raises
``AssertionError`` when the oracle disagrees with a closed form, a brute-force
enumeration, an invariant or a library routine. ``test_oracle_pins.py`` runs
them on the real oracle; ``test_oracle_mutants.py`` runs them on oracles built
with one planted mistake each and checks that some pin fails.
"""
from __future__ import annotations

import itertools

import numpy as np
import scipy.special
import torch

G = 64


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits_via_f32(v: np.ndarray) -> np.ndarray:
    """torch's float32 -> bf16 (RNE) for values exactly representable in fp32."""
    return bf16_bits(torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16))


def pack_nibbles(Q: np.ndarray) -> np.ndarray:
    """Pack an integer matrix ``[N, K]`` (0..15) into ``[N, K/8]`` words:
    element ``8w + i`` goes to bits ``4i .. 4i+3`` of word ``w``."""
    N, K = Q.shape
    Qw = Q.reshape(N, K // 8, 8).astype(np.uint64)
    words = np.zeros((N, K // 8), np.uint64)
    for i in range(8):
        words |= Qw[:, :, i] << np.uint64(4 * i)
    return words.astype(np.uint32)


def rand_bf16(rng, shape, lo, hi) -> np.ndarray:
    return f64_to_bf16_bits_via_f32(rng.uniform(lo, hi, size=shape).astype(np.float32)
                                    .astype(np.float64))


def rand_expert_set(rng, E, N, K, s_lo=0.005, s_hi=0.02):
    Q = rng.integers(0, 16, size=(E, N, K))
    q = np.stack([pack_nibbles(Q[e]) for e in range(E)])
    s = rand_bf16(rng, (E, N, K // G), s_lo, s_hi)
    b = f64_to_bf16_bits_via_f32(-8.0 * bits_to_f64(s) + rng.normal(0, 1e-3, size=s.shape))
    return q, s, b


# ------------------------------------------------------------------ bf16 ---

def pin_bf16(orc):
    assert orc.bf16_to_f64(0x3F80) == 1.0
    assert orc.bf16_to_f64(0xC000) == -2.0
    assert orc.bf16_to_f64(0x0001) == 2.0 ** -133
    assert orc.bf16_to_f64(0x7F7F) == (2 - 2 ** -7) * 2.0 ** 127
    assert orc.f64_to_bf16(1.0) == 0x3F80
    assert orc.f64_to_bf16(1 + 2 ** -8) == 0x3F80            # tie -> even
    assert orc.f64_to_bf16(1 + 3 * 2 ** -8) == 0x3F82        # tie -> even
    assert orc.f64_to_bf16(1 + 2 ** -8 + 2 ** -30) == 0x3F81  # one rounding step
    assert orc.f64_to_bf16(-0.0) == 0x8000
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(4000) * np.exp(rng.uniform(-30, 30, 4000)))
    v = v.astype(np.float32).astype(np.float64)
    want = f64_to_bf16_bits_via_f32(v)
    got = np.array([orc.f64_to_bf16(x) for x in v], np.uint16)
    assert np.array_equal(got, want)


# ------------------------------------------------------------- dequant ---

def pin_dequant_integer(orc):
    rng = np.random.default_rng(2)
    N, K = 24, 192
    Q = rng.integers(0, 16, size=(N, K))
    ones = np.full((N, K // G), 0x3F80, np.uint16)
    zeros = np.zeros((N, K // G), np.uint16)
    W = orc.dequant(pack_nibbles(Q), ones, zeros, G)
    assert np.array_equal(W, Q.astype(np.float64))


def pin_dequant_bias_only(orc):
    rng = np.random.default_rng(3)
    N, K = 16, 256
    b = rand_bf16(rng, (N, K // G), -1.0, 1.0)
    s = rand_bf16(rng, (N, K // G), 0.5, 2.0)
    W = orc.dequant(np.zeros((N, K // 8), np.uint32), s, b, G)
    assert np.array_equal(W, np.repeat(bits_to_f64(b), G, axis=1))


def pin_dequant_one_hot(orc):
    # a single nonzero nibble: W is the bias everywhere except one element
    N, K = 8, 128
    Q = np.zeros((N, K), np.int64)
    Q[5, 77] = 11
    s = np.full((N, K // G), orc.f64_to_bf16(0.25), np.uint16)
    b = np.zeros((N, K // G), np.uint16)
    W = orc.dequant(pack_nibbles(Q), s, b, G)
    want = np.zeros((N, K))
    want[5, 77] = 11 * 0.25
    assert np.array_equal(W, want)


# ------------------------------------------------------------- router ---

def pin_router_library(orc):
    rng = np.random.default_rng(4)
    T, H, E = 5, 96, 12
    x = rand_bf16(rng, (T, H), -2, 2)
    wr = rand_bf16(rng, (H, E), -0.05, 0.05)
    bias = rng.uniform(-3, 3, E).astype(np.float32)
    got = orc.router_logits(x, wr, bias)
    want = bits_to_f64(x) @ bits_to_f64(wr) + bias.astype(np.float64)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    got0 = orc.router_logits(x, wr, None)
    assert np.allclose(got0, bits_to_f64(x) @ bits_to_f64(wr), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- top-k ---

def pin_topk_bruteforce(orc):
    rng = np.random.default_rng(5)
    E = 8
    for k in (1, 2, 3):
        L = rng.standard_normal((9, E))
        idx, w, gap = orc.topk(L, k)
        for t in range(L.shape[0]):
            best = max(itertools.combinations(range(E), k), key=lambda c: L[t, list(c)].sum())
            assert set(idx[t].tolist()) == set(best)
            assert list(idx[t]) == sorted(best, key=lambda e: -L[t, e])
            srt = np.sort(L[t])[::-1]
            assert gap[t] == srt[k - 1] - srt[k]
        if k == 1:
            assert np.array_equal(idx[:, 0], np.argmax(L, axis=1))


def pin_topk_ties(orc):
    L = np.zeros((1, 10))
    idx, _, _ = orc.topk(L, 4)
    assert idx[0].tolist() == [0, 1, 2, 3]
    L = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]])
    idx, w, gap = orc.topk(L, 2)
    assert idx[0].tolist() == [1, 2]
    assert np.allclose(w[0], [0.5, 0.5], rtol=0, atol=1e-15)
    assert gap[0] == 0.0


def pin_topk_nan_and_signed_zero(orc):
    # A NaN logit ranks as -inf (below every number, lower index first among
    # equals) and gets weight zero; -0 and +0 tie; all-NaN rows keep valid,
    # distinct indices (their weights are 0/0).
    nan = float("nan")
    L = np.array([[nan, 1.0, 2.0, nan]])
    idx, w, gap = orc.topk(L, 2)
    assert idx[0].tolist() == [2, 1]
    e = np.exp(1.0)
    assert np.allclose(w[0], [e / (e + 1), 1 / (e + 1)], rtol=1e-15, atol=0)
    assert gap[0] == np.inf                      # runner-up is a NaN (-inf)
    idx, w, _ = orc.topk(L, 3)
    assert idx[0].tolist() == [2, 1, 0] and w[0, 2] == 0.0
    idx, w, _ = orc.topk(L, 4)
    assert idx[0].tolist() == [2, 1, 0, 3] and w[0, 3] == 0.0
    L = np.array([[-0.0, 0.0, -0.0, -1.0]])
    idx, w, gap = orc.topk(L, 2)
    assert idx[0].tolist() == [0, 1] and np.array_equal(w[0], [0.5, 0.5]) and gap[0] == 0.0
    idx, w, _ = orc.topk(np.full((1, 5), nan), 3)
    assert idx[0].tolist() == [0, 1, 2] and np.isnan(w).all()


def pin_topk_weights(orc):
    rng = np.random.default_rng(6)
    E = 16
    L = rng.standard_normal((7, E)) * 2
    idx, w, _ = orc.topk(L, E)               # k = E: the full softmax
    want = np.take_along_axis(scipy.special.softmax(L, axis=1), idx.astype(np.int64), axis=1)
    assert np.allclose(w, want, rtol=1e-13, atol=1e-15)
    for k in (2, 5):
        idx, w, _ = orc.topk(L, k)
        p = np.take_along_axis(scipy.special.softmax(L, axis=1), idx.astype(np.int64), axis=1)
        assert np.allclose(w, p / p.sum(axis=1, keepdims=True), rtol=1e-13, atol=1e-15)
        assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert np.all(w > 0) and np.all(np.diff(w, axis=1) <= 0)


# -------------------------------------------------------- routing maps ---

def check_route_invariants(maps: dict, idx: np.ndarray, E: int, BM: int):
    """Properties any correct routing map has (also used on GPU outputs)."""
    T, k = idx.shape
    cnt, off, toff = maps["counts"], maps["offsets"], maps["tile_offsets"]
    perm, inv, bmap, nt = maps["perm"], maps["inv"], maps["block_map"], maps["num_tiles"]
    assert cnt.sum() == T * k
    assert np.array_equal(cnt, np.bincount(idx.reshape(-1), minlength=E))
    assert off[0] == 0 and np.all(np.diff(off) == cnt) and off[E] == T * k
    tiles = (cnt + BM - 1) // BM
    assert toff[0] == 0 and np.all(np.diff(toff) == tiles) and toff[E] == nt
    assert np.array_equal(np.sort(perm), np.arange(T * k))
    assert np.array_equal(inv[perm], np.arange(T * k))
    flat = idx.reshape(-1)
    for e in range(E):
        seg = perm[off[e]:off[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg // k) > 0)           # stable by token
    assert bmap.shape[0] == nt and bmap[:, 2].sum() == T * k
    assert np.all(bmap[:, 2] >= 1) and np.all(bmap[:, 2] <= BM)
    for b in range(nt):
        e, m0, rows = bmap[b]
        assert off[e] <= m0 and m0 + rows <= off[e + 1]
        assert (m0 - off[e]) % BM == 0 and toff[e] + (m0 - off[e]) // BM == b


def random_topk_idx(rng, T, k, E, weights=None):
    return np.stack([rng.choice(E, size=k, replace=False, p=weights) for _ in range(T)]).astype(np.int32)


def pin_route_maps(orc):
    rng = np.random.default_rng(7)
    for (T, k, E, BM) in ((37, 3, 11, 4), (64, 8, 32, 16), (1, 2, 5, 128)):
        zipf = 1.0 / np.arange(1, E + 1) ** 1.1
        idx = random_topk_idx(rng, T, k, E, zipf / zipf.sum())
        m = orc.route_maps(idx, E, BM)
        check_route_invariants(m, idx, E, BM)
        flat = idx.reshape(-1)
        want_perm = np.array(sorted(range(T * k), key=lambda s: (flat[s], s)), np.int32)
        assert np.array_equal(m["perm"], want_perm)
        want_bmap = []
        for e in range(E):
            c = int((flat == e).sum())
            o = int((flat < e).sum())
            for i in range((c + BM - 1) // BM):
                want_bmap.append((e, o + BM * i, min(BM, c - BM * i)))
        assert np.array_equal(m["block_map"], np.array(want_bmap, np.int32).reshape(-1, 3))


# ------------------------------------------------------------- experts ---

def _flip(m):
    """Negate a packed matrix: q*(-s) + (-b) = -(q*s + b)."""
    q, s, b = m
    return q, s ^ np.uint16(0x8000), b ^ np.uint16(0x8000)


def pin_ffn_odd_identity(orc):
    # silu(g) - silu(-g) = g, so ffn(Wg) - ffn(-Wg) = Wd (g * u)
    rng = np.random.default_rng(8)
    E, H, I = 3, 128, 64
    gate = rand_expert_set(rng, E, I, H, 0.02, 0.1)
    up = rand_expert_set(rng, E, I, H)
    down = rand_expert_set(rng, E, H, I)
    x = bits_to_f64(rand_bf16(rng, (H,), -2, 2))
    for e in range(E):
        plus = orc.expert_ffn(x, e, gate, up, down, G)
        minus = orc.expert_ffn(x, e, _flip(gate), up, down, G)
        Wg = orc.dequant(gate[0][e], gate[1][e], gate[2][e], G)
        Wu = orc.dequant(up[0][e], up[1][e], up[2][e], G)
        Wd = orc.dequant(down[0][e], down[1][e], down[2][e], G)
        want = Wd @ ((Wg @ x) * (Wu @ x))
        assert np.allclose(plus - minus, want, rtol=1e-9, atol=1e-9 * np.abs(want).max())


def pin_ffn_zero_gate(orc):
    # silu(0) = 0: a zero gate matrix gives an exactly zero expert output
    rng = np.random.default_rng(9)
    E, H, I = 2, 128, 64
    gate = (np.zeros((E, I, H // 8), np.uint32), np.zeros((E, I, H // G), np.uint16),
            np.zeros((E, I, H // G), np.uint16))
    up = rand_expert_set(rng, E, I, H)
    down = rand_expert_set(rng, E, H, I)
    x = bits_to_f64(rand_bf16(rng, (H,), -2, 2))
    out = orc.expert_ffn(x, 1, gate, up, down, G)
    assert np.all(out == 0.0)


def _layer_inputs(rng, T, H, I, E):
    x = rand_bf16(rng, (T, H), -2, 2)
    wr = rand_bf16(rng, (H, E), -0.05, 0.05)
    routed = {"gate": rand_expert_set(rng, E, I, H), "up": rand_expert_set(rng, E, I, H),
              "down": rand_expert_set(rng, E, H, I)}
    shared = {"gate": rand_expert_set(rng, 1, I, H), "up": rand_expert_set(rng, 1, I, H),
              "down": rand_expert_set(rng, 1, H, I)}
    return x, wr, routed, shared


def pin_layer_k1(orc):
    # top-1 without a shared expert: y is the argmax expert's output
    rng = np.random.default_rng(10)
    T, H, I, E = 4, 128, 64, 5
    x, wr, routed, _ = _layer_inputs(rng, T, H, I, E)
    bias = rng.uniform(-0.5, 0.5, E).astype(np.float32)
    out = orc.moe_rows(x, wr, bias, routed, None, k=1, G=G)
    am = np.argmax(bits_to_f64(x) @ bits_to_f64(wr) + bias.astype(np.float64), axis=1)
    for t in range(T):
        want = orc.expert_ffn(bits_to_f64(x[t]), int(am[t]), routed["gate"], routed["up"],
                              routed["down"], G)
        assert np.array_equal(out["y"][t], want)
        assert out["topk_w"][t, 0] == 1.0


def pin_layer_shared_weight_one(orc):
    # the shared expert enters with weight 1, the routed ones with w_j
    rng = np.random.default_rng(11)
    T, H, I, E, k = 3, 128, 64, 6, 2
    x, wr, routed, shared = _layer_inputs(rng, T, H, I, E)
    with_sh = orc.moe_rows(x, wr, None, routed, shared, k=k, G=G)
    without = orc.moe_rows(x, wr, None, routed, None, k=k, G=G)
    for t in range(T):
        sh = orc.expert_ffn(bits_to_f64(x[t]), 0, shared["gate"], shared["up"], shared["down"], G)
        assert np.allclose(with_sh["y"][t] - without["y"][t], sh, rtol=1e-12,
                           atol=1e-12 * np.abs(sh).max())
        mix = sum(without["topk_w"][t, j] *
                  orc.expert_ffn(bits_to_f64(x[t]), int(without["topk_idx"][t, j]),
                                 routed["gate"], routed["up"], routed["down"], G)
                  for j in range(k))
        assert np.allclose(without["y"][t], mix, rtol=1e-12, atol=1e-12 * np.abs(mix).max())


def pin_residual(orc):
    rng = np.random.default_rng(12)
    x = rand_bf16(rng, (64,), -3, 3)
    assert np.array_equal(orc.residual(x, np.zeros(64), 0.5), x)
    y = rng.standard_normal(64).astype(np.float32).astype(np.float64)
    got = orc.residual(np.zeros(64, np.uint16), y, 1.0)
    assert np.array_equal(got, f64_to_bf16_bits_via_f32(y))


def pin_rmsnorm(orc):
    # constant rows normalise to +-1 (closed form); output mean square is 1
    # up to bf16 rounding; scaling a row by a power of two changes nothing
    c = np.array([orc.f64_to_bf16(v) for v in (3.0, -0.25, 96.0)], np.uint16)
    rows = np.repeat(c[:, None], 64, axis=1)
    out = bits_to_f64(orc.rmsnorm(rows))
    assert np.array_equal(out, np.sign(bits_to_f64(c))[:, None] * np.ones((3, 64)))
    rng = np.random.default_rng(13)
    x = rand_bf16(rng, (6, 512), -5, 5)
    xn = bits_to_f64(orc.rmsnorm(x))
    assert np.allclose(np.mean(xn ** 2, axis=1), 1.0, rtol=0, atol=5e-3)
    assert np.array_equal(np.sign(xn), np.sign(bits_to_f64(x)))
    x4 = f64_to_bf16_bits_via_f32(bits_to_f64(x) * 4.0)
    d = np.abs(bits_to_f64(orc.rmsnorm(x4)) - xn)
    assert np.all(d <= 2.0 ** -7 * np.abs(xn) + 1e-30)


ALL_PINS = [pin_bf16, pin_dequant_integer, pin_dequant_bias_only, pin_dequant_one_hot,
            pin_router_library, pin_topk_bruteforce, pin_topk_ties,
            pin_topk_nan_and_signed_zero, pin_topk_weights,
            pin_route_maps, pin_ffn_odd_identity, pin_ffn_zero_gate, pin_layer_k1,
            pin_layer_shared_weight_one, pin_residual, pin_rmsnorm]
