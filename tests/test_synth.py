"""The seeded generator: determinism, counter independence and the workload
distributions (no GPU)."""
import numpy as np
import torch

from bit_grouped_gemm_gb300 import synth


def test_splitmix_reference_values():
    # SplitMix64 seeded with 0: first outputs published with the algorithm
    # (Vigna's reference implementation, splitmix64.c)
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    got = synth.stream_u64(0, torch.arange(3))
    got = [int(v) & ((1 << 64) - 1) for v in got.tolist()]
    assert got == want


def test_deterministic_and_prefix_stable():
    a = synth.normal_bf16(5, synth.TAG_X, 0, (4, 64))
    b = synth.normal_bf16(5, synth.TAG_X, 0, (8, 64))
    assert torch.equal(a, b[:4])
    c = synth.normal_bf16(6, synth.TAG_X, 0, (4, 64))
    assert not torch.equal(a, c)


def test_distributions():
    x = synth.normal_bf16(1, synth.TAG_X, 0, (256, 1024)).float()
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1) < 0.01
    w = synth.Workload("t", 4, shape=synth.MoEShape(hidden=256, inter=128, num_experts=8))
    q, s, b = synth.w4_matrix(w, 0, "gate", False)
    assert q.shape == (8, 128, 32) and s.shape == (8, 128, 4) and b.shape == s.shape
    nib = np.stack([(q.numpy().view(np.uint32) >> (4 * i)) & 15 for i in range(8)])
    counts = np.bincount(nib.reshape(-1), minlength=16)
    assert counts.min() > 0.9 * counts.mean()
    sf = s.float()
    assert sf.min() >= 0.0049 and sf.max() <= 0.0201   # bf16 rounding of the bounds
    resid = b.float() + 8 * sf
    assert resid.abs().max() < 0.02 and abs(resid.std().item() - 1e-3) < 5e-4


def test_zipf_bias():
    w = synth.standard_workloads()["t512_zipf"]
    b = synth.router_bias(w, 0)
    assert b.dtype == torch.float32 and b.shape == (256,)
    vals = torch.sort(b, descending=True).values.double()
    want = -1.1 * torch.log(torch.arange(1, 257, dtype=torch.float64))
    assert torch.allclose(vals, want.float().double(), atol=1e-6)
    assert synth.router_bias(synth.standard_workloads()["t128_uniform"], 0) is None
