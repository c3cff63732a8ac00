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


def run_forward(shape, inp, flags=0, token_mask=None):
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
    if shape.expert_dtype == "fp8":
        out["x_amax"] = torch.full((1,), -1.0, dtype=torch.float32, device=DEV)
        out["h_amax"] = torch.full((1,), -1.0, dtype=torch.float32, device=DEV)
    ws = m.alloc_workspace(cfg, DEV)
    aux = {n: out[n] for n in out if n != "y"}
    if token_mask is not None:
        aux["token_mask"] = token_mask.to(DEV)
    m.moe_forward(cfg, inp, inp["x"], out["y"], ws, aux=aux)
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


def e4m3_codes_match(got_vals: torch.Tensor, exact: torch.Tensor, atol: float):
    """E4M3 codes written by the device against the oracle's quantization of the same tensor.

    ``exact`` holds the oracle's unrounded scaled values v = fp64(x) * S; the device rounded its
    own fp32 value of v, which differs from v by up to ``atol`` (the device's fp32 error in x,
    times S). Both round to nearest even, so the codes may differ only where v lies within atol
    of a rounding midpoint, and there the two codes must be neighbours. Returns the number of
    such elements."""
    got = got_vals.double().cpu().flatten()
    want = moe_oracle.e4m3_round(moe_oracle.to_fp32(exact)).flatten()
    bad = (got != want).nonzero().flatten()
    v = exact.double().cpu().flatten()[bad]
    mid = (got[bad] + want[bad]) / 2
    dist = (v - mid).abs()
    step = (got[bad] - want[bad]).abs()
    lo = torch.minimum(got[bad].abs(), want[bad].abs())
    # neighbours: the gap is one E4M3 step at the smaller magnitude (2^(e-3), or 2^-9 below 2^-6)
    _, ex = torch.frexp(lo.clamp_min(2.0 ** -9))
    one_step = step <= torch.exp2((ex - 1 - 3).clamp_min(-9).double()) * 1.0000001
    far = dist > atol
    assert not bool(far.any()), (f"{int(far.sum())} of {bad.numel()} differing codes lie away "
                                 f"from a rounding tie (largest distance {float(dist.max()):.3e}, "
                                 f"atol {atol:.1e})")
    assert bool(one_step.all()), "codes differ by more than one step"
    return int(bad.numel())


def near_tie_router(T=512, d=256, E=64, seed=3, dtype=torch.bfloat16):
    """Router inputs (bf16, or fp32 with dtype) built to defeat fp32 logits: duplicated expert
    columns (exact ties, to be broken by the lower index) and columns that differ only in an
    element weighted by 2^-30 (gaps far below fp32 resolution), plus reordered columns."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, d, generator=g)
    x[:, -1] = 2.0 ** -30                           # a tiny coordinate shared by all tokens
    x = x.to(dtype)
    base = torch.randn(d, 8, generator=g) * d ** -0.5
    cols = []
    for e in range(E):
        c = base[:, e % 8].clone()
        if e % 3 == 1:
            c[-1] += 1.0                          # larger by 2^-30 in exact arithmetic
        if e % 5 == 2:
            c[:-1] = c[:-1][torch.randperm(d - 1, generator=g)]
        cols.append(c)
    w = torch.stack(cols, 1).to(dtype)
    return x, w
