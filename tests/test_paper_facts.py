"""Pins of the packed format's storage accounting to figures the pages print
(tests/golden/paper_facts.txt): 4-bit weights in groups of 64 with a bf16
scale and bias per group make a 35e9-parameter model about 19.4 GB, against
about 70 GB in bf16."""
import os

from bit_grouped_gemm_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def facts():
    out = {}
    with open(os.path.join(HERE, "golden", "paper_facts.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                out[k] = float(v)
    return out


def test_bits_per_weight_matches_checkpoint_size(orc):
    f = facts()
    bpw = orc.bits_per_weight(int(f["group_size"]))
    assert bpw == 4 + (f["scale_bits"] + f["bias_bits"]) / f["group_size"] == 4.5
    size_gb = f["total_params"] * bpw / 8 / 1e9
    # the checkpoint also holds unquantised tensors (embeddings, norms), so
    # only agreement to a few percent is expected
    assert abs(size_gb - f["checkpoint_4bit_GB"]) / f["checkpoint_4bit_GB"] < 0.03
    assert abs(f["total_params"] * 2 / 1e9 - f["bf16_weights_GB"]) < 0.5


def test_model_shape_matches_pages():
    f = facts()
    sh = synth.MoEShape()
    assert sh.num_experts == f["routed_experts"]
    assert sh.top_k == f["experts_per_token"]
    assert int(sh.has_shared) == f["shared_experts"]
    assert sh.group_size == f["group_size"]
    assert synth.standard_workloads()["prefill_t4096_l40_zipf"].layers == \
        f["layers_full_attention"] + f["layers_gated_deltanet"]


def test_expert_bytes():
    # 3*H*I weights at 4.5 bits
    sh = synth.MoEShape()
    assert synth.packed_bytes_per_expert(sh) == 3 * sh.hidden * sh.inter * 4.5 / 8 == 1769472
