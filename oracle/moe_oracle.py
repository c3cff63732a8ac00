"""fp64 CPU oracle of the routed mixture-of-experts forward layer.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and its reference arm) may import this
module. The CUDA library (``sparse_expert_router_gb300``) never imports, links
or runs anything here, and nothing here imports from it. The two share only
the seeded input generators of ``moe_workloads``.

The layer, as the pages state it:
  * "Marin 535B-A23B: the half of a training run nobody usually shows you",
    section "What is actually being trained": every layer's MLP is a mixture of
    384 routed experts of width 3,072, eight chosen per token, plus two shared
    experts every token goes through; routed experts run in a 3,072-wide
    latent: each token is projected down, normalised, sent to its experts and
    projected back up after the weighted combine.
  * "Marin Begins Open Training of a 535B-Parameter MoE Model", section 2: the
    same, and the two shared experts process every token independently of the
    routed path; the output is projected back to model width before it is
    combined with the shared path.
  * Teardown, section "The one knob nobody pinned": the router has a weight
    and a bias.
  * Teardown, section "A sphere for every matrix": expert banks are stacked
    [experts, d_in, d_out].

Readings taken where the pages are silent:
  R1 the router reads the block input x (width d);
  R2 routing is the top-k of the EXACT real-valued logits x.W_r + b of the
     stored inputs, ties to the lowest expert index; indices are reported in
     ascending expert order;
  R3 gates are the softmax over the k selected logits (equal to the full
     softmax renormalised over the selection);
  R4 capacity C = ceil(cf * T * k / E), computed in integers from cf = num/den;
     assignments of expert e beyond C, in token order, are dropped, contribute
     nothing, and the other gates are NOT renormalised ("the token skips that
     expert": teardown section "21% to 27% MFU without stopping the run";
     open-training page section 2);
  R5 RMSNorm h = z / sqrt(mean(z^2) + eps) * gamma, no bias;
  R6 experts are SwiGLU: a = silu(h W1) * (h W3), o = a W2, silu(v) = v / (1 + e^-v)
     computed exactly (the July summary records a ~2.6% mismatch caused by an
     approximate fused SwiGLU epilogue);
  R7 shared experts read x and are summed unweighted;
  R8 y = c W_up + sum_s SwiGLU_s(x);
  R15 an optional token mask marks attention-mask padding, which is excluded from dispatch
     (September 14 weekly summary, hero-run epic, #9159; the teardown's run counts padding
     tokens skipped by routing): a padding token is routed but sends no row to any expert,
     takes no capacity, is not a drop, and keeps only its shared-expert output.

All arithmetic is fp64 on exactly promoted inputs (bf16 and fp32 values are
exact in fp64, and so is every product of two of them). Nothing is rounded
to a lower precision anywhere in this module, except where the layer itself
quantizes: the fp8 expert MLP (section "fp8 expert MLP" below) rounds its
activations to E4M3, taking each rounding decision from the fp32 value the
layer quantizes (readings R12-R14).
"""
from __future__ import annotations

import math
from fractions import Fraction
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

F64 = torch.float64
U64 = 2.0 ** -53          # unit roundoff of fp64


def to64(t: torch.Tensor) -> torch.Tensor:
    """Exact promotion of a stored bf16/fp32 tensor to fp64 on the CPU."""
    return t.detach().to(device="cpu").to(F64)


def expert_weight(inp: Dict[str, torch.Tensor], name: str, e: int) -> torch.Tensor:
    """Expert e's weight matrix in fp64: the stored values, times the per-output-column scale
    when the bank is stored as E4M3 with a `<name>_scale` [E, d_out] tensor (exact in fp64)."""
    w = to64(inp[name][e])
    sc = inp.get(name + "_scale")
    if sc is not None:
        w = w * to64(sc[e]).unsqueeze(0)
    return w


# ---------------------------------------------------------------- router ----

def router_logits(x: torch.Tensor, w_router: torch.Tensor,
                  b_router: Optional[torch.Tensor]) -> Tuple[torch.Tensor, torch.Tensor]:
    """Router logits l[t, e] = sum_i x[t, i] W_r[i, e] + b[e] in fp64, and a bound on their error.

    Every product is exact in fp64, so the only error is the summation of d+1
    terms, bounded for any summation order by gamma_{d+1} * sum|terms| with
    gamma_n = n u / (1 - n u). The sum of |x_i||w_i| is bounded above by
    Cauchy-Schwarz, ||x_t||_2 ||w_e||_2, itself inflated for its own rounding.
    """
    x64, w64 = to64(x), to64(w_router)
    T, d = x64.shape
    logits = x64 @ w64
    babs = torch.zeros(w64.shape[1], dtype=F64)
    if b_router is not None:
        b64 = to64(b_router)
        logits = logits + b64
        babs = b64.abs()
    n = d + 1
    gamma = n * U64 / (1.0 - n * U64)
    cs = x64.norm(dim=1, keepdim=True) * w64.norm(dim=0, keepdim=True)
    bound = (2.0 * gamma) * (cs * (1.0 + 1e-12) + babs) + 1e-300
    return logits, bound


def exact_logit(x_row: Sequence[float], w_col: Sequence[float], b: float) -> Fraction:
    """The exact rational value of one logit: sum of exact products plus the bias."""
    acc = Fraction(b)
    for xi, wi in zip(x_row, w_col):
        if xi != 0.0 and wi != 0.0:
            acc += Fraction(xi) * Fraction(wi)
    return acc


def topk_exact(logits: torch.Tensor, bound: torch.Tensor, k: int,
               exact_fn) -> torch.Tensor:
    """Per token, the k experts with the largest exact logits; ties to the lowest index.

    The fp64 logits decide a token unless the k-th selected and some
    unselected expert overlap within their error bounds; then every expert
    that could still enter the top-k gets its exact value from
    ``exact_fn(t, e)`` and the selection is re-taken on exact values.
    Returns idx [T, k] int64 in ascending expert order (reading R2).
    """
    T, E = logits.shape
    # descending by value; a stable sort keeps equal values in ascending index order
    order = torch.sort(logits, dim=1, descending=True, stable=True).indices
    sel = order[:, :k]
    lo = (logits - bound).gather(1, sel).min(dim=1).values
    if k < E:
        hi = (logits + bound).gather(1, order[:, k:]).max(dim=1).values
    else:
        hi = torch.full((T,), -math.inf, dtype=F64)
    out = sel.clone()
    for t in torch.nonzero(lo <= hi).flatten().tolist():
        cand = torch.nonzero(logits[t] + bound[t] >= lo[t]).flatten().tolist()
        vals = {e: exact_fn(t, e) for e in cand}
        ranked = sorted(cand, key=lambda e: (-vals[e], e))
        out[t] = torch.tensor(ranked[:k])
    return torch.sort(out, dim=1).values


def route(x: torch.Tensor, w_router: torch.Tensor, b_router: Optional[torch.Tensor],
          k: int) -> Dict[str, torch.Tensor]:
    """Router: logits, exact top-k indices (ascending), renormalised softmax gates."""
    logits, bound = router_logits(x, w_router, b_router)
    ws = to64(w_router)
    bs = to64(b_router) if b_router is not None else torch.zeros(ws.shape[1], dtype=F64)

    def exact_fn(t: int, e: int) -> Fraction:
        return exact_logit(to64(x[t]).tolist(), ws[:, e].tolist(), float(bs[e]))

    idx = topk_exact(logits, bound, k, exact_fn)
    return {"logits": logits, "bound": bound, "idx": idx, "gate": softmax_gates(logits, idx)}


def softmax_gates(logits: torch.Tensor, idx: torch.Tensor) -> torch.Tensor:
    """g[t, j] = exp(l_j - m) / sum_{j'} exp(l_j' - m) over the k selected logits (reading R3)."""
    sl = logits.gather(1, idx)
    m = sl.max(dim=1, keepdim=True).values
    ex = torch.exp(sl - m)
    return ex / ex.sum(dim=1, keepdim=True)


# -------------------------------------------------------------- dispatch ----

def capacity(T: int, k: int, E: int, cf: Optional[Tuple[int, int]]) -> Optional[int]:
    """Per-expert capacity C = ceil(num * T * k / (den * E)) in integer arithmetic; None = no limit.

    The open-training page, section 2, gives capacity factors of 1.10 and 1.15;
    the September 14 summary records a capacity rounding that could exceed its
    buffer by one row (#9159). The formula is reading R4.
    """
    if cf is None:
        return None
    num, den = cf
    if num <= 0:
        return None
    return -(-(num * T * k) // (den * E))


def dispatch(idx: torch.Tensor, E: int, cap: Optional[int],
             mask: Optional[torch.Tensor] = None) -> Dict[str, torch.Tensor]:
    """Expert counts, capacity clamp, group offsets and the stable permutation.

    counts[e] = number of assignments to e; kept[e] = min(counts[e], C);
    offsets = exclusive prefix sum of kept (E+1 entries). Assignment (t, j) to
    e gets slot offsets[e] + r, r = number of tokens t' < t that chose e, if
    r < C, else slot -1 (dropped). perm[slot] = t * k + j. Rows of one expert
    therefore sit together in ascending token order, as the ragged transport
    delivers them (teardown, section "21% to 27% MFU without stopping the run").

    mask[t] == 0 marks attention-mask padding (reading R15): the token's assignments are not
    dispatched at all. They are not counted, take no rank and no capacity, are not drops,
    and get slot -1.
    """
    T, k = idx.shape
    il = idx.tolist()
    real = [True] * T if mask is None else [bool(v) for v in mask.tolist()]
    counts = [0] * E
    for t, row in enumerate(il):
        if not real[t]:
            continue
        for e in row:
            counts[e] += 1
    kept = [c if cap is None else min(c, cap) for c in counts]
    offsets = [0] * (E + 1)
    for e in range(E):
        offsets[e + 1] = offsets[e] + kept[e]
    seen = [0] * E
    slot_of = [[-1] * k for _ in range(T)]
    perm = [-1] * offsets[E]
    for t in range(T):
        if not real[t]:
            continue
        for j in range(k):
            e = il[t][j]
            r = seen[e]
            seen[e] += 1
            if cap is None or r < cap:
                s = offsets[e] + r
                slot_of[t][j] = s
                perm[s] = t * k + j
    return {
        "counts": torch.tensor(counts, dtype=torch.int64),
        "kept": torch.tensor(kept, dtype=torch.int64),
        "offsets": torch.tensor(offsets, dtype=torch.int64),
        "slot_of": torch.tensor(slot_of, dtype=torch.int64).reshape(T, k),
        "perm": torch.tensor(perm, dtype=torch.int64),
        "n_dropped": torch.tensor(sum(counts) - sum(kept), dtype=torch.int64),
    }


# --------------------------------------------------------------- latent ----

def latent(x: torch.Tensor, w_down: torch.Tensor, gamma: torch.Tensor,
           eps: float) -> Tuple[torch.Tensor, torch.Tensor]:
    """Latent down-projection z = x W_down and RMSNorm h = z / sqrt(mean(z^2) + eps) * gamma (R5)."""
    z = to64(x) @ to64(w_down)
    ms = (z * z).mean(dim=1, keepdim=True)
    h = z / torch.sqrt(ms + eps) * to64(gamma)
    return z, h


# --------------------------------------------------------------- experts ----

def silu(v: torch.Tensor) -> torch.Tensor:
    """silu(v) = v / (1 + exp(-v)), exact fp64 (reading R6)."""
    return v / (1.0 + torch.exp(-v))


def swiglu_mlp(h: torch.Tensor, w1: torch.Tensor, w3: torch.Tensor,
               w2: torch.Tensor) -> torch.Tensor:
    """One SwiGLU expert: (silu(h W1) * (h W3)) W2, all operands fp64."""
    return (silu(h @ w1) * (h @ w3)) @ w2


def swiglu_hidden(h: torch.Tensor, w1: torch.Tensor, w3: torch.Tensor) -> torch.Tensor:
    """The SwiGLU hidden activation silu(h W1) * (h W3)."""
    return silu(h @ w1) * (h @ w3)


def shared_hidden(x: torch.Tensor, w1_s: torch.Tensor, w3_s: torch.Tensor) -> torch.Tensor:
    """Shared experts' hidden activations, concatenated along the feature axis [T, S*F_s]."""
    x64 = to64(x)
    if w1_s.shape[0] == 0:                       # no shared experts
        return torch.zeros((x64.shape[0], 0), dtype=F64)
    return torch.cat([swiglu_hidden(x64, to64(w1_s[s]), to64(w3_s[s]))
                      for s in range(w1_s.shape[0])], dim=1)


def grouped_experts(rows: torch.Tensor, offsets: Sequence[int], w1: torch.Tensor,
                    w3: torch.Tensor, w2: torch.Tensor,
                    fp8: Optional[Dict[str, object]] = None
                    ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Expert MLPs over expert-grouped rows: rows offsets[e]:offsets[e+1] go through expert e.

    Returns (hidden a [R, F], output o [R, L]) in fp64 for the active rows
    only; rows past offsets[-1] (pool padding) are never computed, matching
    the "mask-free" ragged expert MLP of the teardown's section
    "21% to 27% MFU without stopping the run".
    With ``fp8`` (keys w1_scale, w3_scale, w2_scale, x_scale, h_scale) the rows are E4M3
    codes and every expert runs fp8_expert; a is then the hidden before its quantization.
    """
    r64 = to64(rows)
    n_act = int(offsets[-1])
    F = w1.shape[2]
    bank = {"w1": w1, "w3": w3, "w2": w2}
    if fp8:
        bank.update({k: v for k, v in fp8.items() if k.endswith("_scale")})
    a = torch.zeros((n_act, F), dtype=F64)
    o = torch.zeros((n_act, w2.shape[2]), dtype=F64)
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            W1, W3, W2 = (expert_weight(bank, n, e) for n in ("w1", "w3", "w2"))
            if fp8:
                o[lo:hi], a[lo:hi], _ = fp8_expert(r64[lo:hi], float(fp8["x_scale"]),
                                                   float(fp8["h_scale"]), W1, W3, W2)
            else:
                a[lo:hi] = swiglu_hidden(r64[lo:hi], W1, W3)
                o[lo:hi] = a[lo:hi] @ W2
    return a, o


# ------------------------------------------------------------ fp8 expert MLP ----
#
# The July summary (section on the B200 training MFU epic, #6880 and #7079) describes an fp8
# ragged dot for the expert MLP: E4M3 in the forward pass, with delayed scaling (the scale of a
# tensor comes from the amax recorded at earlier steps). Readings taken here:
#   R12 both operands of each expert GEMM are E4M3: the grouped rows x_perm, quantized with the
#       per-tensor multiplier S_x, and the SwiGLU hidden a, quantized with S_h; the expert
#       weights are E4M3 with one scale per output column (weight ~ code * scale);
#   R13 quantization is q = e4m3(fp32(v * S)) (round to nearest even, saturating at 448) and
#       dequantization multiplies by fp32(1 / S); S_x and S_h are inputs (the delayed-scaling
#       state), and the layer reports this step's amax of each quantized tensor;
#   R14 router, latent projection, shared experts, combine and up-projection stay 16-bit.

E4M3_MAX = 448.0


def e4m3_round(v: torch.Tensor) -> torch.Tensor:
    """Nearest E4M3 value of each element (fp64 in, fp64 out), ties to the even code;
    magnitudes above the largest finite value, 448, saturate to it.

    E4M3 has a sign, 4 exponent bits (bias 7) and 3 fraction bits: normal values
    1.f x 2^e for e in [-6, 8] (the all-ones code of e = 8 is NaN, so 1.75 x 2^8 = 448 is the
    largest finite value) and subnormal values 0.f x 2^-6. Within [2^e, 2^(e+1)) consecutive
    values are 2^(e-3) apart; below 2^-6 they are 2^-9 apart. Rounding to the nearest multiple
    of that step, ties to the even multiple, is round-to-nearest-even on the code."""
    v = to64(v)
    a = v.abs()
    _, ex = torch.frexp(a)                      # a = m * 2^ex with m in [0.5, 1)
    e = torch.clamp(ex - 1, min=-6)             # binade of a; the subnormal range uses e = -6
    step = torch.exp2((e - 3).to(F64))
    r = torch.clamp(torch.round(a / step) * step, max=E4M3_MAX)   # torch.round: half to even
    return torch.sign(v) * r


def to_fp32(v: torch.Tensor) -> torch.Tensor:
    """Round to the nearest fp32 value (as fp64)."""
    return to64(v).to(torch.float32).to(F64)


def quantize_e4m3(v: torch.Tensor, scale: float) -> torch.Tensor:
    """E4M3 codes (as their values) of v under the quantization multiplier `scale` (R13):
    e4m3(fp32(v * scale)). The product is rounded to fp32 first, the precision in which the
    layer holds the activations it quantizes, so that both roundings decide as the layer does."""
    return e4m3_round(to_fp32(to64(v) * float(scale)))


def dequant_multiplier(scale: float) -> float:
    """fp32(1 / scale), correctly rounded (numpy's fp32 division is IEEE)."""
    return float(np.float32(1.0) / np.float32(scale))


def fp8_expert(codes: torch.Tensor, x_scale: float, h_scale: float, w1: torch.Tensor,
               w3: torch.Tensor, w2: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor,
                                                          torch.Tensor]:
    """One expert's fp8 forward on rows already quantized to E4M3 codes (R12, R13):
    xq = codes * fp32(1/S_x); a = silu(xq W1) * (xq W3); aq = e4m3(fp32(a S_h)) * fp32(1/S_h);
    o = aq W2, with W* the dequantized weights. Returns (o, a, the codes of a)."""
    xq = to64(codes) * dequant_multiplier(x_scale)
    a = swiglu_hidden(xq, w1, w3)
    a_codes = quantize_e4m3(a, h_scale)
    o = (a_codes * dequant_multiplier(h_scale)) @ w2
    return o, a, a_codes


def combine(y_perm: torch.Tensor, slot_of: torch.Tensor, gate: torch.Tensor) -> torch.Tensor:
    """c[t] = sum over kept j, in ascending expert order, of gate[t, j] * y_perm[slot_of[t, j]].

    A dropped assignment (slot -1) contributes nothing and the other gates are
    not renormalised (reading R4). The fixed j order is the ordered-gather
    combine that made repeated scoring bitwise exact (September 14 summary,
    post-training epic, #9144).
    """
    yp = to64(y_perm)
    g = to64(gate)
    T, k = slot_of.shape
    c = torch.zeros((T, yp.shape[1]), dtype=F64)
    for j in range(k):
        s = slot_of[:, j]
        keep = s >= 0
        if keep.any():
            c[keep] += g[keep, j:j + 1] * yp[s[keep]]
    return c


# -------------------------------------------------------- expert MLP backward ----
#
# The July summary (#5330, the Grug MoE microbenchmark) moves the backward of the ragged dot to a
# custom VJP: the input gradient is a grouped GEMM against the transposed expert weights, and the
# weight gradient a GEMM that contracts over each expert's ragged rows. Written out for the
# SwiGLU expert MLP y = (silu(x W1) * (x W3)) W2 by the chain rule.

def silu_grad(v: torch.Tensor) -> torch.Tensor:
    """d silu(v) / dv = s (1 + v (1 - s)) with s = 1 / (1 + e^-v), fp64."""
    s = 1.0 / (1.0 + torch.exp(-v))
    return s * (1.0 + v * (1.0 - s))


def grouped_experts_backward(rows: torch.Tensor, offsets: Sequence[int], w1: torch.Tensor,
                             w3: torch.Tensor, w2: torch.Tensor, dy: torch.Tensor, *,
                             weight_grads: bool = True) -> Dict[str, torch.Tensor]:
    """Gradients of the grouped expert MLP (grouped_experts) given dy = dL/dy_perm.

    For expert e with rows X = rows[offsets[e]:offsets[e+1]], G = X W1_e, U = X W3_e,
    A = silu(G) * U (the forward's hidden) and Y = A W2_e:
      dA = dY W2_e^T,  dG = dA * U * silu'(G),  dU = dA * silu(G),
      dX = dG W1_e^T + dU W3_e^T,
      dW1_e = X^T dG,  dW3_e = X^T dU,  dW2_e = A^T dY.
    Experts without rows get zero weight gradients; rows past offsets[-1] get no dX. All fp64.
    Returns dx [n_active, L], dw1, dw3 [E, L, F], dw2 [E, F, L] and the intermediates
    g, u, a, da, dg, du [n_active, F]. With weight_grads=False the three weight gradients are
    neither formed nor returned (a check of dx alone on a large expert bank)."""
    x64, dy64 = to64(rows), to64(dy)
    n_act = int(offsets[-1])
    E, L, F = w1.shape
    out = {"dx": torch.zeros((n_act, L), dtype=F64)}
    if weight_grads:
        out.update({"dw1": torch.zeros((E, L, F), dtype=F64),
                    "dw3": torch.zeros((E, L, F), dtype=F64),
                    "dw2": torch.zeros((E, F, w2.shape[2]), dtype=F64)})
    for n in ("g", "u", "a", "da", "dg", "du"):
        out[n] = torch.zeros((n_act, F), dtype=F64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi <= lo:
            continue
        X, dY = x64[lo:hi], dy64[lo:hi]
        W1, W3, W2 = to64(w1[e]), to64(w3[e]), to64(w2[e])
        G, U = X @ W1, X @ W3
        A = silu(G) * U
        dA = dY @ W2.T
        dG = dA * U * silu_grad(G)
        dU = dA * silu(G)
        out["dx"][lo:hi] = dG @ W1.T + dU @ W3.T
        if weight_grads:
            out["dw1"][e] = X.T @ dG
            out["dw3"][e] = X.T @ dU
            out["dw2"][e] = A.T @ dY
        for n, v in (("g", G), ("u", U), ("a", A), ("da", dA), ("dg", dG), ("du", dU)):
            out[n][lo:hi] = v
    return out


# --------------------------------------------------------------- forward ----

def forward(inp: Dict[str, torch.Tensor], *, top_k: int, rms_eps: float,
            capacity_factor: Optional[Tuple[int, int]] = None,
            tokens: Optional[Sequence[int]] = None) -> Dict[str, torch.Tensor]:
    """The whole layer: route, dispatch, latent, experts, combine, up-projection + shared.

    An optional ``inp["token_mask"]`` [T] marks padding tokens with 0 (reading R15): they are
    routed like every token but not dispatched, so their routed part c[t] is zero and
    y[t] is the shared experts' output alone.

    Routing and dispatch are always computed for every token (capacity drops
    depend on all earlier tokens). The expert, combine and output stages are
    computed for ``tokens`` only when given (each token's output depends only
    on its own row and its own routing), else for all tokens.
    Returned tensors for those stages are indexed by position in ``tokens``.
    """
    x = inp["x"]
    T = x.shape[0]
    E = inp["w_router"].shape[1]
    r = route(x, inp["w_router"], inp.get("b_router"), top_k)
    cap = capacity(T, top_k, E, capacity_factor)
    dsp = dispatch(r["idx"], E, cap, inp.get("token_mask"))
    toks = list(range(T)) if tokens is None else [int(t) for t in tokens]
    xt = x[toks]
    z, h = latent(xt, inp["w_down"], inp["rms_gamma"], rms_eps)
    w1, w3, w2 = inp["w1"], inp["w3"], inp["w2"]
    L = w2.shape[2]
    idx = r["idx"][toks]
    slot = dsp["slot_of"][toks]
    gate = r["gate"][toks]
    # per assignment expert output o[t, j] (zero when dropped)
    o = torch.zeros((len(toks), top_k, L), dtype=F64)
    by_expert: Dict[int, List[Tuple[int, int]]] = {}
    for i in range(len(toks)):
        for j in range(top_k):
            if int(slot[i, j]) >= 0:
                by_expert.setdefault(int(idx[i, j]), []).append((i, j))
    fp8 = "x_scale" in inp
    amax_x = amax_h = 0.0
    for e in sorted(by_expert):
        pairs = by_expert[e]
        rows = torch.stack([h[i] for i, _ in pairs])
        W1, W3, W2 = (expert_weight(inp, n, e) for n in ("w1", "w3", "w2"))
        if fp8:
            sx, sh = float(inp["x_scale"].reshape(-1)[0]), float(inp["h_scale"].reshape(-1)[0])
            out_e, a_e, _ = fp8_expert(quantize_e4m3(rows, sx), sx, sh, W1, W3, W2)
            amax_x = max(amax_x, float(rows.abs().max()))
            amax_h = max(amax_h, float(a_e.abs().max()))
        else:
            out_e = swiglu_mlp(rows, W1, W3, W2)
        for n, (i, j) in enumerate(pairs):
            o[i, j] = out_e[n]
    c = torch.zeros((len(toks), L), dtype=F64)
    for j in range(top_k):
        kept = slot[:, j] >= 0
        c[kept] += gate[kept, j:j + 1] * o[kept, j]
    a_s = shared_hidden(xt, inp["w1_s"], inp["w3_s"])
    w2s = to64(inp["w2_s"]).reshape(-1, to64(inp["w2_s"]).shape[-1])
    y = c @ to64(inp["w_up"]) + a_s @ w2s
    out = dict(r)
    out.update(dsp)
    out.update({"tokens": torch.tensor(toks, dtype=torch.int64), "z": z, "h": h, "o": o,
                "c": c, "a_s": a_s, "y": y, "capacity": torch.tensor(-1 if cap is None else cap)})
    if fp8:   # amax of the tensors the layer quantized, over the computed tokens' kept rows
        out.update({"x_amax": torch.tensor(amax_x, dtype=F64),
                    "h_amax": torch.tensor(amax_h, dtype=F64)})
    return out


# --------------------------------------------------------------- layer backward ----

def backward(inp: Dict[str, torch.Tensor], fwd: Dict[str, torch.Tensor], dy: torch.Tensor, *,
             rms_eps: float, expert_weight_grads: bool = True) -> Dict[str, torch.Tensor]:
    """Gradients of <dy, y> for the whole layer (16-bit or fp32 expert banks), by the chain
    rule through the forward's definition, given ``fwd`` = forward(inp, ...) over all tokens.

    Top-k selection is piecewise constant, so no gradient flows through the choice of experts;
    it flows through the selected logits' softmax gates. With G = the selected gates and dG the
    gradient of the gates, the selected logits get G_j (dG_j - sum_i G_i dG_i).
      y = c W_up + a_s W2s                  -> dc = dy W_up^T, dW_up = c^T dy, da_s = dy W2s^T,
                                               dW2s = a_s^T dy
      c[t] = sum_j g[t,j] o[t,j] (kept j)   -> do[t,j] = g[t,j] dc[t], dg[t,j] = <dc[t], o[t,j]>
      o = expert MLP of h (per expert)      -> grouped_experts_backward
      h = z rstd gamma, rstd = (mean(z^2) + eps)^-1/2
                                            -> dgamma = sum_t dh z rstd,
                                               dz = rstd (dh gamma - zhat mean(dh gamma zhat))
      z = x W_down                          -> dW_down = x^T dz, dx += dz W_down^T
      logits = x W_r + b                    -> dW_r = x^T dl, db = sum_t dl, dx += dl W_r^T
      shared: a_s = silu(x W1_s) (x W3_s)   -> as the expert MLP, dx += ...
    Returns every gradient in fp64 (names d<weight>, dx). expert_weight_grads=False leaves out
    dw1, dw3 and dw2 of the routed experts (whose fp64 banks would be 87 GB for the 535B layer);
    everything else, dx included, is unchanged."""
    x64, dy64 = to64(inp["x"]), to64(dy)
    T, d = x64.shape
    E = inp["w_router"].shape[1]
    k = fwd["idx"].shape[1]
    L = inp["w_up"].shape[0]
    idx, gate, slot = fwd["idx"], fwd["gate"], fwd["slot_of"]
    w_up = to64(inp["w_up"])
    w2s = to64(inp["w2_s"])
    S, Fs = w2s.shape[0], w2s.shape[1]
    out: Dict[str, torch.Tensor] = {}
    # up-projection and the shared experts' down projection
    dc = dy64 @ w_up.T
    out["dw_up"] = fwd["c"].T @ dy64
    da_s = dy64 @ w2s.reshape(S * Fs, d).T
    out["dw2_s"] = (fwd["a_s"].T @ dy64).reshape(S, Fs, d)
    # shared experts (read x)
    dx = torch.zeros((T, d), dtype=F64)
    out["dw1_s"] = torch.zeros_like(to64(inp["w1_s"]))
    out["dw3_s"] = torch.zeros_like(to64(inp["w3_s"]))
    for s in range(S):
        W1, W3 = to64(inp["w1_s"][s]), to64(inp["w3_s"][s])
        G, U = x64 @ W1, x64 @ W3
        dA = da_s[:, s * Fs:(s + 1) * Fs]
        dG = dA * U * silu_grad(G)
        dU = dA * silu(G)
        out["dw1_s"][s] = x64.T @ dG
        out["dw3_s"][s] = x64.T @ dU
        dx += dG @ W1.T + dU @ W3.T
    # combine: per kept assignment
    o = fwd["o"]
    dgate = torch.zeros((T, k), dtype=F64)
    kept = slot >= 0
    dgate[kept] = (dc.unsqueeze(1) * o).sum(-1)[kept]
    # expert MLPs over the kept assignments in dispatch order (rows of expert e by token)
    E_rows: Dict[int, List[Tuple[int, int]]] = {}
    for t in range(T):
        for j in range(k):
            if int(slot[t, j]) >= 0:
                E_rows.setdefault(int(idx[t, j]), []).append((t, j))
    h = fwd["h"]
    order = [(e, t, j) for e in sorted(E_rows) for (t, j) in E_rows[e]]
    offsets = [0] * (E + 1)
    for e in range(E):
        offsets[e + 1] = offsets[e] + len(E_rows.get(e, []))
    rows = torch.stack([h[t] for _, t, _ in order]) if order else torch.zeros((0, L), dtype=F64)
    dys = (torch.stack([gate[t, j] * dc[t] for _, t, j in order]) if order
           else torch.zeros((0, L), dtype=F64))
    eb = grouped_experts_backward(rows, offsets, inp["w1"], inp["w3"], inp["w2"], dys,
                                  weight_grads=expert_weight_grads)
    if expert_weight_grads:
        out["dw1"], out["dw3"], out["dw2"] = eb["dw1"], eb["dw3"], eb["dw2"]
    dh = torch.zeros((T, L), dtype=F64)
    for n, (_, t, _) in enumerate(order):
        dh[t] += eb["dx"][n]
    # RMSNorm and the down-projection
    z = fwd["z"]
    rstd = 1.0 / torch.sqrt((z * z).mean(dim=1, keepdim=True) + rms_eps)
    zhat = z * rstd
    gamma = to64(inp["rms_gamma"])
    out["drms_gamma"] = (dh * zhat).sum(0)
    dhg = dh * gamma
    dz = rstd * (dhg - zhat * (dhg * zhat).mean(dim=1, keepdim=True))
    out["dw_down"] = x64.T @ dz
    dx += dz @ to64(inp["w_down"]).T
    # router: softmax over the selected logits
    dl = torch.zeros((T, E), dtype=F64)
    s_t = (gate * dgate).sum(1, keepdim=True)
    dsel = gate * (dgate - s_t)
    for j in range(k):
        dl[torch.arange(T), idx[:, j]] += dsel[:, j]
    out["dw_router"] = x64.T @ dl
    out["db_router"] = dl.sum(0)
    dx += dl @ to64(inp["w_router"]).T
    out["dx"] = dx
    out["dgate"] = dgate
    out["dh"] = dh
    return out


def slice_forward(inp: Dict[str, torch.Tensor]) -> Dict[str, torch.Tensor]:
    """One expert-parallel rank's slice: grouped SwiGLU experts over the pool, then the
    gate-weighted un-permute back to arrival order: out[i] = gate[i] * o[slot_of[i]]."""
    offs = [int(v) for v in inp["expert_offsets"].tolist()]
    a, o = grouped_experts(inp["pool"], offs, inp["w1"], inp["w3"], inp["w2"])
    s = inp["slot_of"].to(torch.int64)
    out = to64(inp["gate"]).unsqueeze(1) * o[s]
    return {"a": a, "y_perm": o, "out": out}


def slice_rows(inp: Dict[str, torch.Tensor], positions: Sequence[int]) -> Dict[str, torch.Tensor]:
    """The slice workload for selected arrival positions only (each row is independent):
    for position i, pool row r = slot_of[i] of expert e (offsets[e] <= r < offsets[e+1]),
    o = SwiGLU_e(pool[r]) and out[i] = gate[i] * o."""
    offs = [int(v) for v in inp["expert_offsets"].tolist()]
    pos = [int(p) for p in positions]
    rows = [int(inp["slot_of"][p]) for p in pos]
    groups: Dict[int, List[int]] = {}
    for n, r in enumerate(rows):
        e = max(g for g in range(len(offs) - 1) if offs[g] <= r < offs[g + 1])
        groups.setdefault(e, []).append(n)
    L = inp["w2"].shape[2]
    o = torch.zeros((len(pos), L), dtype=F64)
    for e, ns in groups.items():
        v = to64(inp["pool"][[rows[n] for n in ns]])
        o[ns] = swiglu_mlp(v, expert_weight(inp, "w1", e), expert_weight(inp, "w3", e),
                           expert_weight(inp, "w2", e))
    g = to64(inp["gate"][pos]).unsqueeze(1)
    return {"rows": torch.tensor(rows), "y_perm": o, "out": g * o}
