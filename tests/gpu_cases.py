"""Helpers of the GPU parity tests: run the CUDA library through its C ABI and the fp64
oracle on the same seeded inputs, and compare."""
import torch

import sparse_expert_router_gb300 as m
from moe_workloads import make_layer_inputs
from oracle import moe_oracle

DEV = "cuda"


def normwise(a: torch.Tensor, b: torch.Tensor) -> float:
    """||a - b||_F / ||b||_F in fp64."""
    a = a.detach().double().cpu()
    b = b.detach().double().cpu()
    return float((a - b).norm() / b.norm().clamp_min(1e-300))


def gpu_inputs(shape):
    """Seeded inputs drawn on the GPU (large shapes) or on the CPU and copied (small ones)."""
    if shape.T * shape.d_model >= (1 << 24) or shape.n_experts * shape.d_ff * shape.d_latent >= (1 << 27):
        return make_layer_inputs(shape, DEV)
    return {k: v.to(DEV) for k, v in make_layer_inputs(shape, "cpu").items()}


def run_forward(shape, inp, flags=0):
    cfg = m.LayerConfig.from_shape(shape, flags=flags)
    T, k, E = shape.T, shape.top_k, shape.n_experts
    out = {
        "y": torch.empty((T, shape.d_model), dtype=shape.torch_dtype, device=DEV),
        "topk_idx": torch.full((T, k), -7, dtype=torch.int32, device=DEV),
        "topk_gate": torch.zeros((T, k), dtype=torch.float32, device=DEV),
        "expert_counts": torch.zeros(E, dtype=torch.int32, device=DEV),
        "expert_offsets": torch.zeros(E + 1, dtype=torch.int32, device=DEV),
        "slot_of": torch.zeros((T, k), dtype=torch.int32, device=DEV),
        "n_dropped": torch.zeros(1, dtype=torch.int32, device=DEV),
    }
    ws = m.alloc_workspace(cfg, DEV)
    m.moe_forward(cfg, inp, inp["x"], out["y"], ws, aux={n: out[n] for n in out if n != "y"})
    out["report"] = m.moe_get_device_status(ws)
    out["ws"] = ws
    return out


def sample_tokens(T, n, seed=0, extra=()):
    g = torch.Generator().manual_seed(seed)
    base = torch.randperm(T, generator=g)[:n].tolist()
    return sorted(set(base) | set(int(t) for t in extra))


def oracle_forward(shape, inp, tokens=None):
    return moe_oracle.forward(inp, top_k=shape.top_k, rms_eps=shape.rms_eps,
                              capacity_factor=shape.capacity, tokens=tokens)


def check_routing(got, ref, shape):
    """Bit-exact routing and dispatch; gates within the fp32 tolerance."""
    assert torch.equal(got["topk_idx"].cpu().long(), ref["idx"]), "top-k indices differ"
    gtol = 1e-6 if shape.dtype == "f32" else 1e-5
    gerr = float((got["topk_gate"].cpu().double() - ref["gate"]).abs().max())
    assert gerr <= gtol, f"gate error {gerr}"
    assert torch.equal(got["expert_counts"].cpu().long(), ref["counts"])
    assert torch.equal(got["expert_offsets"].cpu().long(), ref["offsets"])
    assert torch.equal(got["slot_of"].cpu().long(), ref["slot_of"])
    assert int(got["n_dropped"].cpu()) == int(ref["n_dropped"])
    return gerr
