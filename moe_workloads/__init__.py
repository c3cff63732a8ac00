"""Seeded synthetic workloads for the routed-MoE forward layer.

This module holds shapes and seeded random-number draws only: it contains none
of the layer's arithmetic. Both the fp64 oracle (``oracle/``) and the CUDA
library's tests and benchmark consume the tensors it makes, so that the two
sides see identical stored inputs.

Shapes follow the layer the Marin pages describe (384 routed experts, top-8,
two shared experts, width 6,144 with a normalised 3,072-wide latent:
"Marin 535B-A23B: the half of a training run nobody usually shows you",
section "What is actually being trained"; "Marin Begins Open Training of a
535B-Parameter MoE Model", section 2). The smaller shapes are scaled-down
members of the same family.

Recipe (stated once, used everywhere):
  * x ~ N(0, 1); every weight ~ N(0, 1/fan_in) with fan_in = d_in of that
    matrix; RMSNorm gain = 1; router bias = 0 ("near-uniform routing": with
    W_r ~ N(0, 1/d) the logits are about N(0, 1) and i.i.d. over experts).
  * Values are drawn in fp32 by torch's seeded generator, scaled, then rounded
    to the config dtype with round-to-nearest-even.
  * Every tensor has its own generator, seeded from (seed, tensor id, leading
    index), so tensors are independent of one another and of generation order.
  * Zipf-skewed routing adds a fixed bias b[e] = -beta * s * ln(rank(e)) to the
    router logits, rank = a seeded permutation of 1..E (Zipf popularity
    p ~ rank^-s; the normaliser of p cancels in top-k and in the gates).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass
from typing import Dict, Optional, Tuple

import numpy as np
import torch

__all__ = [
    "LayerShape", "SliceShape", "SHAPES", "SLICE_C5B", "get_shape",
    "make_layer_inputs", "make_slice_inputs", "ZIPF_BETA", "zipf_bias",
    "tensor_seed", "make_router_inputs",
]

# Scale of the log-popularity bias. 1.0 means the logits are biased by ln(p_e)
# itself, the plain reading of "router logits biased by a Zipf(s=1.1) expert
# popularity". At seed 0 and T=16384 on the 535B-shaped layer the hottest
# expert then gets 46x the mean load (the top-8 ceiling is 48x) and 162 of 384
# experts get no token. Smaller scales that bring the hottest expert near 20x
# the mean leave no expert empty.
ZIPF_BETA = 1.0


@dataclass(frozen=True)
class LayerShape:
    """One routed-MoE layer workload: sizes, precision, routing recipe."""

    name: str
    T: int                 # tokens
    d_model: int           # model width d
    d_latent: int          # latent width L
    n_experts: int         # routed experts E
    top_k: int             # experts per token k
    d_ff: int              # routed expert SwiGLU width F
    n_shared: int          # shared experts S
    d_ff_shared: int       # shared expert SwiGLU width F_s
    dtype: str             # "f32" or "bf16"
    capacity: Optional[Tuple[int, int]] = None   # capacity factor as (num, den); None = no drop
    routing: str = "uniform"                     # "uniform" or "zipf"
    zipf_s: float = 1.1
    seed: int = 0
    rms_eps: float = 1e-6
    expert_dtype: str = "bf16"   # routed expert banks: "bf16", or "fp8" (E4M3 + per-column scales)
    # fp8 experts: per-tensor quantization multipliers of the grouped rows and of the SwiGLU
    # hidden (the delayed-scaling state). Powers of two that keep the largest expected values
    # (|rows| <= ~7 after the RMSNorm, |hidden| <= ~30) below the E4M3 maximum of 448.
    fp8_x_scale: float = 32.0
    fp8_h_scale: float = 8.0

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_(self, **kw) -> "LayerShape":
        return dataclasses.replace(self, **kw)

    def flops(self) -> Dict[str, float]:
        """Algorithmic multiply-add work (2 flops each) per stage of one forward."""
        T, d, L, E, k = self.T, self.d_model, self.d_latent, self.n_experts, self.top_k
        F, SF = self.d_ff, self.n_shared * self.d_ff_shared
        R = T * k
        return {
            "router": 2.0 * T * d * E,
            "down": 2.0 * T * d * L,
            "shared_up": 2.0 * T * d * 2 * SF,
            "expert_up": 2.0 * R * L * 2 * F,
            "expert_down": 2.0 * R * F * L,
            "back": 2.0 * T * (L + SF) * d,
        }


@dataclass(frozen=True)
class SliceShape:
    """One expert-parallel rank's compute slice: pre-grouped rows, grouped GEMMs + un-permute."""

    name: str
    rows: int              # active rows that arrive
    pool_rows: int         # physical rows of the fixed receive pool (padding at the end)
    d_latent: int
    n_local: int           # local experts
    d_ff: int
    alpha: float           # Dirichlet concentration of the expert shares
    seed: int = 0
    dtype: str = "bf16"


SHAPES: Dict[str, LayerShape] = {
    # Tiny fp32 layer: every stage checked in full against the oracle in seconds.
    "tiny_f32": LayerShape("tiny_f32", T=256, d_model=256, d_latent=128, n_experts=16,
                           top_k=2, d_ff=128, n_shared=1, d_ff_shared=256, dtype="f32"),
    # Small bf16 layer.
    "small_bf16": LayerShape("small_bf16", T=4096, d_model=2048, d_latent=1024, n_experts=64,
                             top_k=8, d_ff=1024, n_shared=2, d_ff_shared=2048, dtype="bf16"),
    # 535B-shaped layer, one 8,192-token batch.
    "l535b_t8192": LayerShape("l535b_t8192", T=8192, d_model=6144, d_latent=3072, n_experts=384,
                              top_k=8, d_ff=3072, n_shared=2, d_ff_shared=3072, dtype="bf16"),
    # Same layer, Zipf(1.1)-skewed expert popularity, no drop and capacity factor 1.10.
    "l535b_zipf_t16384": LayerShape("l535b_zipf_t16384", T=16384, d_model=6144, d_latent=3072,
                                    n_experts=384, top_k=8, d_ff=3072, n_shared=2,
                                    d_ff_shared=3072, dtype="bf16", routing="zipf"),
    "l535b_zipf_t16384_cf110": LayerShape("l535b_zipf_t16384_cf110", T=16384, d_model=6144,
                                          d_latent=3072, n_experts=384, top_k=8, d_ff=3072,
                                          n_shared=2, d_ff_shared=3072, dtype="bf16",
                                          routing="zipf", capacity=(11, 10)),
    # Long context: one 65,536-token sequence through the full layer.
    "l535b_t65536": LayerShape("l535b_t65536", T=65536, d_model=6144, d_latent=3072,
                               n_experts=384, top_k=8, d_ff=3072, n_shared=2, d_ff_shared=3072,
                               dtype="bf16"),
    # Profiling case (a few GB on the device): the 535B layer's widths with 64 of its 384
    # experts and T=1368, so each expert gets ~171 rows, the same as at T=8192 with all experts.
    "l535b_e64_t1368": LayerShape("l535b_e64_t1368", T=1368, d_model=6144, d_latent=3072,
                                  n_experts=64, top_k=8, d_ff=3072, n_shared=2,
                                  d_ff_shared=3072, dtype="bf16"),
    # Profiling case of the routing, dispatch and combine kernels (2.5 GB on the device): the
    # 535B layer at T=8192 with the routed experts' d_ff cut to 128. Router, dispatch and combine
    # see exactly the bench workload's sizes (T, d, latent, E, k), and their inputs exceed L2.
    "l535b_f128_t8192": LayerShape("l535b_f128_t8192", T=8192, d_model=6144, d_latent=3072,
                                   n_experts=384, top_k=8, d_ff=128, n_shared=2,
                                   d_ff_shared=3072, dtype="bf16"),
}

# fp8 expert weights (E4M3 with a power-of-two scale per expert output column), everything
# else as the bf16 shapes above.
SHAPES["small_fp8"] = SHAPES["small_bf16"].with_(name="small_fp8", expert_dtype="fp8")
SHAPES["l535b_t8192_fp8"] = SHAPES["l535b_t8192"].with_(name="l535b_t8192_fp8", expert_dtype="fp8")
SHAPES["l535b_e64_t1368_fp8"] = SHAPES["l535b_e64_t1368"].with_(name="l535b_e64_t1368_fp8",
                                                                expert_dtype="fp8")

# One GPU of a 64-way expert-parallel domain: 6 local experts, 49,152 arriving
# latent rows, receive pool sized with the receiver capacity factor 1.15 and
# rounded up to a multiple of 128 rows.
SLICE_C5B = SliceShape("l535b_ep_slice", rows=49152, pool_rows=56576, d_latent=3072,
                       n_local=6, d_ff=3072, alpha=0.5)

# Stable ids that key each tensor's generator.
_TENSOR_IDS = {
    "x": 1, "w_router": 2, "w_down": 3, "w1": 4, "w3": 5, "w2": 6, "w1_s": 7, "w3_s": 8,
    "w2_s": 9, "w_up": 10, "zipf_perm": 11, "slice_x": 12, "slice_w1": 13, "slice_w3": 14,
    "slice_w2": 15, "slice_draws": 16, "padding_mask": 17,
}


def get_shape(name: str) -> LayerShape:
    return SHAPES[name]


def tensor_seed(seed: int, tensor: str, index: int = 0) -> int:
    """Seed of one tensor's generator (or of one leading slice of it)."""
    tid = _TENSOR_IDS[tensor]
    return (seed * 0x9E3779B1 + tid * 0x85EBCA77 + index * 0xC2B2AE3D + 0x165667B1) % (1 << 63)


def _normal(shape, std: float, dtype: torch.dtype, device, seed: int) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _stacked_normal(n: int, rows: int, cols: int, std: float, dtype, device, seed: int,
                    tensor: str) -> torch.Tensor:
    """[n, rows, cols] weights, slice i drawn by its own generator (bounded fp32 temporaries)."""
    out = torch.empty((n, rows, cols), dtype=dtype, device=device)
    for i in range(n):
        out[i].copy_(_normal((rows, cols), std, dtype, device, tensor_seed(seed, tensor, i)))
    return out


FP8_MAX = 448.0   # largest finite E4M3 value


def _stacked_fp8(n: int, rows: int, cols: int, std: float, device, seed: int, tensor: str):
    """[n, rows, cols] E4M3 weights and [n, cols] fp32 scales: slice i is drawn like
    _stacked_normal (fp32), each column is divided by the power of two that brings its largest
    magnitude to at most 448, and rounded to E4M3 (nearest even). The layer's weight is the
    E4M3 value times its column's scale."""
    q = torch.empty((n, rows, cols), dtype=torch.float8_e4m3fn, device=device)
    sc = torch.empty((n, cols), dtype=torch.float32, device=device)
    for i in range(n):
        w = _normal((rows, cols), std, torch.float32, device, tensor_seed(seed, tensor, i))
        amax = w.abs().amax(dim=0).clamp_min(1e-30)
        scale = torch.exp2(torch.ceil(torch.log2(amax / FP8_MAX)))
        q[i].copy_((w / scale).to(torch.float8_e4m3fn))
        sc[i].copy_(scale)
    return q, sc


def zipf_bias(shape: LayerShape, beta: float = ZIPF_BETA) -> torch.Tensor:
    """Router bias giving a Zipf(s) expert popularity: b[e] = -beta * s * ln(rank(e))."""
    g = torch.Generator(device="cpu")
    g.manual_seed(tensor_seed(shape.seed, "zipf_perm"))
    rank = torch.randperm(shape.n_experts, generator=g).to(torch.float64) + 1.0
    return (-beta * shape.zipf_s * torch.log(rank)).to(torch.float32)


def make_layer_inputs(shape: LayerShape, device="cpu", *, T: Optional[int] = None,
                      zipf_beta: float = ZIPF_BETA) -> Dict[str, torch.Tensor]:
    """All inputs of one layer forward: activations x and every weight.

    Layouts (row-major): x [T, d]; w_router [d, E]; b_router [E] fp32;
    w_down [d, L]; rms_gamma [L] fp32; w1, w3 [E, L, F]; w2 [E, F, L] (with
    expert_dtype "fp8": E4M3, plus w1_scale, w3_scale [E, F] and w2_scale [E, L] fp32, and the
    activation quantization multipliers x_scale, h_scale [1] fp32);
    w1_s, w3_s [S, d, F_s]; w2_s [S, F_s, d]; w_up [L, d].
    Expert banks are stacked [experts, d_in, d_out] as the teardown's
    section "A sphere for every matrix" describes.
    """
    s = shape
    T = s.T if T is None else T
    dt = s.torch_dtype
    d, L, E, F, S, Fs = s.d_model, s.d_latent, s.n_experts, s.d_ff, s.n_shared, s.d_ff_shared
    out = {
        "x": _normal((T, d), 1.0, dt, device, tensor_seed(s.seed, "x")),
        "w_router": _normal((d, E), d ** -0.5, dt, device, tensor_seed(s.seed, "w_router")),
        "w_down": _normal((d, L), d ** -0.5, dt, device, tensor_seed(s.seed, "w_down")),
        "rms_gamma": torch.ones(L, dtype=torch.float32, device=device),
        "w1_s": _stacked_normal(S, d, Fs, d ** -0.5, dt, device, s.seed, "w1_s"),
        "w3_s": _stacked_normal(S, d, Fs, d ** -0.5, dt, device, s.seed, "w3_s"),
        "w2_s": _stacked_normal(S, Fs, d, max(Fs, 1) ** -0.5, dt, device, s.seed, "w2_s"),
        "w_up": _normal((L, d), L ** -0.5, dt, device, tensor_seed(s.seed, "w_up")),
    }
    if s.expert_dtype == "fp8":
        out["x_scale"] = torch.tensor([s.fp8_x_scale], dtype=torch.float32, device=device)
        out["h_scale"] = torch.tensor([s.fp8_h_scale], dtype=torch.float32, device=device)
        out["w1"], out["w1_scale"] = _stacked_fp8(E, L, F, L ** -0.5, device, s.seed, "w1")
        out["w3"], out["w3_scale"] = _stacked_fp8(E, L, F, L ** -0.5, device, s.seed, "w3")
        out["w2"], out["w2_scale"] = _stacked_fp8(E, F, L, F ** -0.5, device, s.seed, "w2")
    else:
        out["w1"] = _stacked_normal(E, L, F, L ** -0.5, dt, device, s.seed, "w1")
        out["w3"] = _stacked_normal(E, L, F, L ** -0.5, dt, device, s.seed, "w3")
        out["w2"] = _stacked_normal(E, F, L, F ** -0.5, dt, device, s.seed, "w2")
    if s.routing == "zipf":
        out["b_router"] = zipf_bias(s, zipf_beta).to(device)
    else:
        out["b_router"] = torch.zeros(E, dtype=torch.float32, device=device)
    return out


def make_slice_inputs(sh: SliceShape, device="cpu") -> Dict[str, torch.Tensor]:
    """Inputs of the expert-parallel slice workload.

    Returns pool [pool_rows, L] (active rows grouped by local expert at the
    front, zero padding rows after them), expert_offsets [E+1] int32 (group
    boundaries of the active rows), gate [rows] fp32 in (0, 1], slot_of [rows]
    int32 (pool row of each arrival position), and the local experts' w1, w3
    [E, L, F] and w2 [E, F, L].
    """
    rng = np.random.Generator(np.random.Philox(tensor_seed(sh.seed, "slice_draws")))
    shares = rng.dirichlet([sh.alpha] * sh.n_local)
    counts = rng.multinomial(sh.rows, shares)
    offsets = np.zeros(sh.n_local + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    gate = (1.0 - rng.random(sh.rows)).astype(np.float32)        # U(0, 1]
    ret = rng.permutation(sh.rows)                                # pool row r returns to position ret[r]
    slot_of = np.empty(sh.rows, dtype=np.int64)
    slot_of[ret] = np.arange(sh.rows)
    dt = torch.bfloat16 if sh.dtype == "bf16" else torch.float32
    L, F, E = sh.d_latent, sh.d_ff, sh.n_local
    pool = torch.zeros((sh.pool_rows, L), dtype=dt, device=device)
    pool[: sh.rows].copy_(_normal((sh.rows, L), 1.0, dt, device, tensor_seed(sh.seed, "slice_x")))
    return {
        "pool": pool,
        "expert_offsets": torch.from_numpy(offsets.astype(np.int32)).to(device),
        "gate": torch.from_numpy(gate).to(device),
        "slot_of": torch.from_numpy(slot_of.astype(np.int32)).to(device),
        "w1": _stacked_normal(E, L, F, L ** -0.5, dt, device, sh.seed, "slice_w1"),
        "w3": _stacked_normal(E, L, F, L ** -0.5, dt, device, sh.seed, "slice_w3"),
        "w2": _stacked_normal(E, F, L, F ** -0.5, dt, device, sh.seed, "slice_w2"),
    }


def make_router_inputs(shape: LayerShape, device="cpu") -> Dict[str, torch.Tensor]:
    """Only the router's inputs (x, w_router, b_router) of make_layer_inputs(shape, device),
    drawn identically, without the expert weights."""
    s = shape
    dt = s.torch_dtype
    out = {
        "x": _normal((s.T, s.d_model), 1.0, dt, device, tensor_seed(s.seed, "x")),
        "w_router": _normal((s.d_model, s.n_experts), s.d_model ** -0.5, dt, device,
                            tensor_seed(s.seed, "w_router")),
    }
    if s.routing == "zipf":
        out["b_router"] = zipf_bias(s).to(device)
    else:
        out["b_router"] = torch.zeros(s.n_experts, dtype=torch.float32, device=device)
    return out


def padding_mask(T: int, seq_len: int = 64, max_pad_frac: float = 0.5, seed: int = 0,
                 device="cpu") -> torch.Tensor:
    """[T] uint8 attention mask of packed sequences: the tokens are cut into sequences of
    `seq_len`, and each sequence ends with a seeded run of padding (0) of up to
    `max_pad_frac` of its length; real tokens are 1."""
    g = torch.Generator().manual_seed(tensor_seed(seed, "padding_mask"))
    mask = torch.ones(T, dtype=torch.uint8)
    for s0 in range(0, T, seq_len):
        n = min(seq_len, T - s0)
        pad = int(torch.randint(0, int(n * max_pad_frac) + 1, (1,), generator=g))
        if pad:
            mask[s0 + n - pad:s0 + n] = 0
    return mask.to(device)
