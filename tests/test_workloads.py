"""The seeded input generators: deterministic, independent per tensor, right shapes (CPU)."""
import torch

from moe_workloads import SHAPES, SLICE_C5B, make_layer_inputs, make_slice_inputs, zipf_bias


def test_layer_inputs_deterministic_and_shaped():
    s = SHAPES["tiny_f32"]
    a = make_layer_inputs(s)
    b = make_layer_inputs(s)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    assert a["x"].shape == (s.T, s.d_model) and a["x"].dtype == torch.float32
    assert a["w1"].shape == (s.n_experts, s.d_latent, s.d_ff)
    assert a["w2"].shape == (s.n_experts, s.d_ff, s.d_latent)
    assert a["w1_s"].shape == (s.n_shared, s.d_model, s.d_ff_shared)
    assert a["w2_s"].shape == (s.n_shared, s.d_ff_shared, s.d_model)
    assert not torch.equal(a["w1"], a["w3"])
    # N(0, 1/fan_in): the empirical std of a large matrix is close to fan_in^-1/2
    assert abs(float(a["w_up"].float().std()) * s.d_latent ** 0.5 - 1.0) < 0.05


def test_bf16_rounding_and_seed():
    s = SHAPES["small_bf16"].with_(T=64)
    a = make_layer_inputs(s)
    assert a["x"].dtype == torch.bfloat16 and a["b_router"].dtype == torch.float32
    c = make_layer_inputs(s.with_(seed=1))
    assert not torch.equal(a["x"], c["x"])


def test_zipf_bias_is_log_popularity():
    s = SHAPES["l535b_zipf_t16384"]
    b = zipf_bias(s, 1.0).double()
    rank = torch.argsort(torch.argsort(-b)) + 1          # rank 1 = most popular
    assert torch.allclose(b, -1.1 * torch.log(rank.double()), atol=1e-5)


def test_slice_inputs():
    sh = SLICE_C5B.__class__(**{**SLICE_C5B.__dict__, "rows": 1000, "pool_rows": 1152, "d_latent": 64, "d_ff": 32})
    d = make_slice_inputs(sh)
    off = d["expert_offsets"].tolist()
    assert off[0] == 0 and off[-1] == 1000 and all(a <= b for a, b in zip(off, off[1:]))
    assert sorted(d["slot_of"].tolist()) == list(range(1000))
    assert float(d["gate"].min()) > 0.0 and float(d["gate"].max()) <= 1.0
    assert d["pool"][1000:].abs().sum() == 0


def test_fp8_expert_weights():
    s = SHAPES["small_fp8"].with_(T=32, n_experts=8, d_latent=64, d_ff=32)
    a = make_layer_inputs(s)
    assert a["w1"].dtype == torch.float8_e4m3fn and a["w1_scale"].shape == (8, 32)
    assert a["w2_scale"].shape == (8, 64)
    sc = a["w1_scale"]
    assert torch.equal(torch.exp2(torch.log2(sc).round()), sc)          # powers of two
    deq = a["w1"].float() * sc.unsqueeze(1)
    assert float(deq.abs().amax(dim=1).div(sc).max()) <= 448.0
    # the dequantized weights stay close to the bf16 draw of the same generator
    ref = make_layer_inputs(s.with_(expert_dtype="bf16"))["w1"].float()
    assert float((deq - ref).norm() / ref.norm()) < 0.05
