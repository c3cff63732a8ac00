"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than the oracle itself:
brute-force enumeration, closed forms, hand-derived fixtures under
tests/golden/, invariants of the layer, and an independently written dense
pipeline. test_planted_mistakes_are_caught plants plausible mistakes in the
oracle (on the CPU) and shows that some pin fails for each.
"""
import itertools
import json
import math
import os

import pytest
import torch
import torch.nn.functional as Fn

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F64 = torch.float64


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand_layer(T=24, d=12, L=8, E=6, F=5, S=2, Fs=7, seed=0, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s, sc=1.0: (torch.randn(*s, generator=g) * sc).to(dtype)
    return {
        "x": r(T, d), "w_router": r(d, E, sc=d ** -0.5), "b_router": torch.zeros(E),
        "w_down": r(d, L, sc=d ** -0.5), "rms_gamma": (1.0 + 0.1 * torch.randn(L, generator=g)),
        "w1": r(E, L, F, sc=L ** -0.5), "w3": r(E, L, F, sc=L ** -0.5), "w2": r(E, F, L, sc=F ** -0.5),
        "w1_s": r(S, d, Fs, sc=d ** -0.5), "w3_s": r(S, d, Fs, sc=d ** -0.5),
        "w2_s": r(S, Fs, d, sc=Fs ** -0.5), "w_up": r(L, d, sc=L ** -0.5),
    }


# ------------------------------------------------------------ pin functions ----
# Written as plain functions so that the planted-mistake test can re-run them.

def pin_topk_bruteforce(seed=0):
    """Top-k with ties to the lowest index == the max-sum k-subset, ties to the
    lexicographically smallest sorted tuple, enumerated over all C(E, k) subsets.
    Integer-valued inputs make exact integer logits with many ties."""
    g = torch.Generator().manual_seed(seed)
    for (E, k, d) in [(16, 2, 5), (10, 3, 4), (8, 1, 3), (7, 7, 3), (12, 4, 2)]:
        x = torch.randint(-2, 3, (12, d), generator=g).float()
        w = torch.randint(-1, 2, (d, E), generator=g).float()
        b = torch.randint(-1, 2, (E,), generator=g).float()
        got = O.route(x, w, b, k)["idx"]
        xi, wi, bi = x.long().tolist(), w.long().tolist(), b.long().tolist()
        for t in range(x.shape[0]):
            logit = [sum(xi[t][i] * wi[i][e] for i in range(d)) + bi[e] for e in range(E)]
            best = max(itertools.combinations(range(E), k),
                       key=lambda c: (sum(logit[e] for e in c), [-e for e in c]))
            assert got[t].tolist() == list(best), (E, k, t, logit, got[t].tolist(), best)


def pin_topk_exact_near_tie():
    """Two experts whose exact logits differ by far less than fp64 resolves: the
    exact value must decide, and a true tie must go to the lower index."""
    d = 6
    x = torch.tensor([[1.0, 1.0, 1.0, 1.0, 1.0, 2.0 ** -60]], dtype=torch.float32)
    base = torch.tensor([0.5, -0.25, 0.125, 1.0, 0.75, 0.0])
    cols = []
    for e in range(5):
        cols.append(base - 4.0 * (e + 1))        # clearly smaller experts
    hi_a = base.clone()
    hi_b = base.clone()
    hi_b[5] = 1.0                                 # exact logit larger by 2^-60
    w = torch.stack([hi_a] + cols + [hi_b], dim=1).float()   # expert 0 = a, expert 6 = b
    idx = O.route(x, w, None, 1)["idx"]
    assert idx.tolist() == [[6]], idx
    w2 = torch.stack([hi_a] + cols + [hi_a], dim=1).float()  # exact tie: lower index wins
    assert O.route(x, w2, None, 1)["idx"].tolist() == [[0]]
    _ = d


def pin_logit_bound_holds(seed=1):
    """The fp64 logit error stays inside the oracle's bound (exact values by rationals)."""
    lay = _rand_layer(T=6, d=40, E=5, seed=seed, dtype=torch.bfloat16)
    logits, bound = O.router_logits(lay["x"], lay["w_router"], lay["b_router"])
    xs, ws = O.to64(lay["x"]), O.to64(lay["w_router"])
    for t in range(6):
        for e in range(5):
            ex = O.exact_logit(xs[t].tolist(), ws[:, e].tolist(), 0.0)
            assert abs(float(ex - __import__("fractions").Fraction(float(logits[t, e])))) <= float(bound[t, e])


def pin_gates():
    """Gates sum to 1; for k=2 they are sigmoid(l1 - l2); they equal the full softmax
    renormalised over the selected experts."""
    lay = _rand_layer(T=32, d=16, E=9, seed=3)
    for k in (1, 2, 4):
        r = O.route(lay["x"], lay["w_router"], lay["b_router"], k)
        g = r["gate"]
        assert torch.allclose(g.sum(1), torch.ones(32, dtype=F64), atol=1e-15, rtol=0)
        full = torch.softmax(r["logits"], dim=1).gather(1, r["idx"])
        assert torch.allclose(g, full / full.sum(1, keepdim=True), atol=1e-15, rtol=0)
        if k == 1:
            assert torch.equal(g, torch.ones_like(g))
        if k == 2:
            l = r["logits"].gather(1, r["idx"])
            assert torch.allclose(g[:, 0], torch.sigmoid(l[:, 0] - l[:, 1]), atol=1e-15, rtol=0)


def pin_capacity():
    """Integer ceiling of cf*T*k/E; a float product would overshoot by one row."""
    assert O.capacity(16384, 8, 384, (11, 10)) == 376           # ceil(375.47)
    assert O.capacity(50, 1, 1, (11, 10)) == 55                 # 1.1*50 in floats is 55.00000000000001
    assert O.capacity(100, 8, 8, (11, 10)) == 110               # 1.1*100 in floats is 110.00000000000001
    assert O.capacity(100, 1, 10, (1, 1)) == 10
    assert O.capacity(7, 2, 3, (1, 1)) == 5                     # ceil(14/3)
    assert O.capacity(5, 2, 3, None) is None
    assert O.capacity(5, 2, 3, (0, 1)) is None


def pin_dispatch_golden():
    gd = _load("dispatch_capacity.json")
    idx = torch.tensor(gd["idx"])
    cap = O.capacity(idx.shape[0], idx.shape[1], gd["n_experts"], tuple(gd["capacity_factor"]))
    assert cap == gd["expected_capacity"]
    d = O.dispatch(idx, gd["n_experts"], cap)
    assert d["counts"].tolist() == gd["expected_counts"]
    assert d["kept"].tolist() == gd["expected_kept"]
    assert d["offsets"].tolist() == gd["expected_offsets"]
    assert d["slot_of"].tolist() == gd["expected_slot_of"]
    assert d["perm"].tolist() == gd["expected_perm"]
    assert int(d["n_dropped"]) == gd["expected_n_dropped"]


def pin_dispatch_invariants(seed=5):
    """Counts sum to T*k; slots are a bijection onto [0, sum kept); perm inverts slot_of;
    within an expert slots ascend with t; the dropped assignments are exactly those past
    capacity in token order (checked against a sort-based recomputation)."""
    g = torch.Generator().manual_seed(seed)
    T, E, k = 200, 11, 3
    idx = torch.stack([torch.randperm(E, generator=g)[:k].sort().values for _ in range(T)])
    for cap in (None, 40, 55, 1):
        d = O.dispatch(idx, E, cap)
        assert int(d["counts"].sum()) == T * k
        slots = d["slot_of"].flatten()
        kept = slots[slots >= 0]
        assert sorted(kept.tolist()) == list(range(int(d["kept"].sum())))
        for t in range(T):
            for j in range(k):
                s = int(d["slot_of"][t, j])
                if s >= 0:
                    assert int(d["perm"][s]) == t * k + j
        # sort-based: all assignments ordered by (expert, token)
        order = sorted(((int(idx[t, j]), t, j) for t in range(T) for j in range(k)))
        pos, rank = 0, {}
        for e, t, j in order:
            rank[(t, j)] = sum(1 for (e2, t2, _) in order if e2 == e and t2 < t)
        off = d["offsets"].tolist()
        for e, t, j in order:
            r = rank[(t, j)]
            exp = off[e] + r if (cap is None or r < cap) else -1
            assert int(d["slot_of"][t, j]) == exp
            pos += 1
        assert int(d["n_dropped"]) == int((slots < 0).sum())


def _dense_pipeline(lay, e, eps):
    """An independently written dense layer: up(SwiGLU_e(RMSNorm(down(x)))) + shared(x)."""
    x = lay["x"].double()
    z = torch.einsum("td,dl->tl", x, lay["w_down"].double())
    h = z * torch.rsqrt(z.pow(2).mean(-1, keepdim=True) + eps) * lay["rms_gamma"].double()
    hid = Fn.silu(torch.einsum("tl,lf->tf", h, lay["w1"][e].double())) * \
        torch.einsum("tl,lf->tf", h, lay["w3"][e].double())
    routed = torch.einsum("tf,fl->tl", hid, lay["w2"][e].double())
    y = torch.einsum("tl,ld->td", routed, lay["w_up"].double())
    for s in range(lay["w1_s"].shape[0]):
        hs = Fn.silu(x @ lay["w1_s"][s].double()) * (x @ lay["w3_s"][s].double())
        y = y + hs @ lay["w2_s"][s].double()
    return y


def pin_forced_single_expert():
    """k=1 and a +1e4 bias on one expert: every gate is 1 and the layer equals a dense MLP."""
    for e_star in (0, 4):
        lay = _rand_layer(T=20, seed=11 + e_star)
        lay["b_router"] = torch.zeros(6)
        lay["b_router"][e_star] = 1e4
        out = O.forward(lay, top_k=1, rms_eps=1e-6)
        assert (out["idx"] == e_star).all()
        ref = _dense_pipeline(lay, e_star, 1e-6)
        err = (out["y"] - ref).norm() / ref.norm()
        assert err <= 1e-12, float(err)


def pin_identical_experts():
    """All routed experts equal and no drop: gates sum to 1, so the output does not depend
    on the routing and equals the dense pipeline with that one expert."""
    lay = _rand_layer(T=16, seed=21)
    for name in ("w1", "w3", "w2"):
        lay[name] = lay[name][:1].expand_as(lay[name]).clone()
    for k in (2, 3):
        out = O.forward(lay, top_k=k, rms_eps=1e-6)
        ref = _dense_pipeline(lay, 0, 1e-6)
        assert ((out["y"] - ref).norm() / ref.norm()) <= 1e-12


def pin_two_token_golden():
    gd = _load("two_token_layer.json")
    lay = {kk: torch.tensor(gd[kk], dtype=torch.float32) for kk in
           ("x", "w_router", "b_router", "w_down", "rms_gamma", "w1", "w3", "w2", "w1_s",
            "w3_s", "w2_s", "w_up")}
    out = O.forward(lay, top_k=gd["top_k"], rms_eps=gd["rms_eps"])
    assert out["idx"].tolist() == gd["expected_idx"]
    env = {"sig": lambda v: 1.0 / (1.0 + math.exp(-v)), "sqrt": math.sqrt}
    exp = torch.tensor([[eval(s, {"__builtins__": {}}, env) for s in row]
                        for row in gd["expected_y"]], dtype=F64)
    assert torch.allclose(out["y"], exp, atol=1e-14, rtol=0), (out["y"], exp)


def pin_rmsnorm():
    """With gamma = 1 and eps = 0, mean(h^2) = 1 and h is invariant to scaling z by c > 0."""
    g = torch.Generator().manual_seed(4)
    x = torch.randn(10, 12, generator=g)
    w = torch.randn(12, 8, generator=g)
    _, h = O.latent(x, w, torch.ones(8), 0.0)
    assert torch.allclose((h * h).mean(1), torch.ones(10, dtype=F64), atol=1e-14, rtol=0)
    _, h2 = O.latent(x * 4.0, w, torch.ones(8), 0.0)
    assert torch.allclose(h, h2, atol=1e-14, rtol=0)


def pin_combine_drop_not_renormalised():
    """A dropped assignment contributes nothing and the kept gates keep their values."""
    yp = torch.tensor([[1.0, 2.0], [10.0, 20.0]])
    slot = torch.tensor([[0, -1], [1, 0]])
    gate = torch.tensor([[0.25, 0.75], [0.5, 0.5]])
    c = O.combine(yp, slot, gate)
    assert c.tolist() == [[0.25, 0.5], [5.5, 11.0]]


def _tiny_slice(seed=9):
    g = torch.Generator().manual_seed(seed)
    E, L, F, P = 3, 6, 5, 14
    offs = [0, 4, 4, 10]                      # an empty expert; rows 10..13 are padding
    inp = {"pool": torch.randn(P, L, generator=g), "expert_offsets": torch.tensor(offs),
           "w1": torch.randn(E, L, F, generator=g), "w3": torch.randn(E, L, F, generator=g),
           "w2": torch.randn(E, F, L, generator=g),
           "gate": torch.rand(10, generator=g), "slot_of": torch.randperm(10, generator=g)}
    inp["pool"][10:] = float("nan")           # padding must never be read
    return inp, offs


def _slice_row_by_hand(inp, offs, i):
    """Arrival position i by hand: its pool row, that row's expert (the group whose half-open
    range holds it), SwiGLU, gate."""
    r = int(inp["slot_of"][i])
    e = [ee for ee in range(len(offs) - 1) if offs[ee] <= r < offs[ee + 1]]
    assert len(e) == 1
    v = inp["pool"][r].double()
    W1, W3, W2 = (inp[n][e[0]].double() for n in ("w1", "w3", "w2"))
    return float(inp["gate"][i]) * ((Fn.silu(v @ W1) * (v @ W3)) @ W2)


def pin_slice_rowwise():
    """The grouped slice, whole (slice_forward) and for chosen positions (slice_rows), equals a
    per-row loop that looks up each row's expert; rows at group boundaries (pool rows 0, 3, 4
    and 9, next to the empty expert) are among the positions."""
    inp, offs = _tiny_slice()
    out = O.slice_forward(inp)["out"]
    assert not bool(torch.isnan(out).any())
    # the positions whose pool rows sit at group boundaries, in no particular order
    pos = [int((inp["slot_of"] == r).nonzero()) for r in (4, 0, 9, 3, 6)]
    part = O.slice_rows(inp, pos)
    assert part["rows"].tolist() == [4, 0, 9, 3, 6]
    for i in range(10):
        ref = _slice_row_by_hand(inp, offs, i)
        assert torch.allclose(out[i], ref, atol=1e-12, rtol=0)
    for n, i in enumerate(pos):
        ref = _slice_row_by_hand(inp, offs, i)
        assert torch.allclose(part["out"][n], ref, atol=1e-12, rtol=0), (i, n)
        r = int(inp["slot_of"][i])
        assert torch.allclose(part["y_perm"][n] * float(inp["gate"][i]), ref, atol=1e-12, rtol=0)
        assert torch.equal(part["y_perm"][n], O.slice_forward(inp)["y_perm"][r])


def pin_forward_drop_skips_expert():
    """With a capacity, each dropped assignment removes exactly gate * expert output from
    the token's routed sum; kept gates are unchanged (the token skips that expert)."""
    lay = _rand_layer(T=40, E=4, seed=31)
    k = 2
    full = O.forward(lay, top_k=k, rms_eps=1e-6)
    capd = O.forward(lay, top_k=k, rms_eps=1e-6, capacity_factor=(1, 2))   # C = 10 of ~20 per expert
    assert int(capd["n_dropped"]) > 0
    x = lay["x"].double()
    z = x @ lay["w_down"].double()
    h = z * torch.rsqrt(z.pow(2).mean(-1, keepdim=True) + 1e-6) * lay["rms_gamma"].double()
    for t in range(40):
        diff = full["y"][t] - capd["y"][t]
        exp = torch.zeros_like(diff)
        for j in range(k):
            if int(capd["slot_of"][t, j]) < 0:
                e = int(full["idx"][t, j])
                hid = Fn.silu(h[t] @ lay["w1"][e].double()) * (h[t] @ lay["w3"][e].double())
                exp += float(full["gate"][t, j]) * ((hid @ lay["w2"][e].double()) @ lay["w_up"].double())
        assert torch.allclose(diff, exp, atol=1e-12, rtol=0), t


def pin_fp8_expert_golden():
    """fp8 expert MLP (E4M3 weights with column scales, E4M3 rows and hidden under per-tensor
    multipliers), hand-derived from the E4M3 value grid."""
    gd = _load("fp8_expert_scales.json")
    lay = {kk: torch.tensor(gd[kk], dtype=torch.float32) for kk in
           ("x", "w_router", "b_router", "w_down", "rms_gamma", "w1_s", "w3_s", "w2_s", "w_up")}
    for n in ("w1", "w3", "w2"):
        lay[n] = torch.tensor(gd[n + "_fp8"], dtype=torch.float32).to(torch.float8_e4m3fn)
        lay[n + "_scale"] = torch.tensor(gd[n + "_scale"], dtype=torch.float32)
    lay["x_scale"] = torch.tensor([gd["x_scale"]], dtype=torch.float32)
    lay["h_scale"] = torch.tensor([gd["h_scale"]], dtype=torch.float32)
    out = O.forward(lay, top_k=gd["top_k"], rms_eps=gd["rms_eps"])
    assert torch.equal(out["y"], torch.tensor(gd["expected_y"], dtype=F64)), out["y"]
    env = {"sig": lambda v: 1.0 / (1.0 + math.exp(-v)), "sqrt": math.sqrt}
    for key in ("x_amax", "h_amax"):
        want = eval(gd["expected_" + key], {"__builtins__": {}}, env)
        assert abs(float(out[key]) - want) <= 1e-15 * want, (key, float(out[key]), want)


def _e4m3_table():
    """Every finite E4M3 value with its code, decoded by torch's float8_e4m3fn type."""
    codes = torch.arange(256, dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(F64)
    fin = ~torch.isnan(vals)
    return codes[fin].long(), vals[fin]


def _nearest_even_bruteforce(v: torch.Tensor) -> torch.Tensor:
    """Nearest finite E4M3 value by search over the whole decoded table; at equal distance the
    value whose code is even; beyond 448 the largest magnitude of the sign (saturation)."""
    codes, vals = _e4m3_table()
    out = torch.empty_like(v)
    for i, x in enumerate(v.tolist()):
        if abs(x) >= 448.0:
            out[i] = math.copysign(448.0, x)
            continue
        d = (vals - x).abs()
        best = d.min()
        cand = (d == best).nonzero().flatten()
        if len(cand) > 1:
            even = [c for c in cand.tolist() if int(codes[c]) % 2 == 0]
            cand = torch.tensor(even or cand.tolist())
        out[i] = vals[int(cand[0])]
    return out


def pin_e4m3_rounding():
    """E4M3 rounding against a brute-force search of the value table, and against torch's own
    float8 conversion of fp32 values in range: exact ties, both sides of every tie, every value,
    subnormals and saturation."""
    _, vals = _e4m3_table()
    pos = torch.unique(vals[vals > 0])
    mids = (pos[1:] + pos[:-1]) / 2                               # exact ties
    g = torch.Generator().manual_seed(11)
    rnd = torch.randn(400, generator=g, dtype=F64) * torch.exp2(
        torch.randint(-12, 9, (400,), generator=g).to(F64))
    probe = torch.cat([pos, mids, mids * (1 + 2.0 ** -30), mids * (1 - 2.0 ** -30), rnd,
                       torch.tensor([0.0, 2.0 ** -10, 3 * 2.0 ** -11, 449.0, 464.0, 479.9,
                                     480.0, 1e6])])
    probe = torch.cat([probe, -probe])
    got = O.e4m3_round(probe)
    assert torch.equal(got, _nearest_even_bruteforce(probe))
    # torch converts through fp32 (then to nearest even): compare on fp32 values
    p32 = O.to_fp32(probe[probe.abs() <= 448.0])
    lib = p32.to(torch.float32).to(torch.float8_e4m3fn).to(F64)
    assert torch.equal(O.e4m3_round(p32), lib)
    assert float(O.e4m3_round(torch.tensor([464.0]))) == 448.0
    assert float(O.e4m3_round(torch.tensor([1.0625]))) == 1.0      # tie to even code
    assert float(O.e4m3_round(torch.tensor([1.1875]))) == 1.25     # tie to even code


def pin_fp8_quantize_in_fp32():
    """The rounding decision is taken on the fp32 product: 1.0625 + 2^-40 is an E4M3 tie once
    rounded to fp32 (to even: 1.0), though nearer to 1.125 in exact arithmetic."""
    v = torch.tensor([1.0625 + 2.0 ** -40], dtype=F64)
    assert float(O.quantize_e4m3(v, 1.0)) == 1.0
    assert float(O.quantize_e4m3(v * 2, 0.5)) == 1.0
    assert O.dequant_multiplier(3.0) == float(torch.tensor(1 / 3, dtype=torch.float32))


def pin_fp8_layer_grid():
    """On a small random fp8 layer every quantized row and hidden value the oracle produces is
    the brute-force nearest E4M3 value of its fp32-rounded scaled input."""
    from moe_workloads import SHAPES, make_layer_inputs
    s = SHAPES["small_fp8"].with_(T=24, d_model=64, n_experts=8, d_latent=32, d_ff=32,
                                  n_shared=1, d_ff_shared=32)
    inp = make_layer_inputs(s, "cpu")
    out = O.forward(inp, top_k=s.top_k, rms_eps=s.rms_eps)
    sx, sh = float(inp["x_scale"][0]), float(inp["h_scale"][0])
    e = int(out["idx"][0, 0])
    rows = out["h"][(out["idx"] == e).any(1)]
    codes = O.quantize_e4m3(rows, sx)
    flat = O.to_fp32(rows * sx).flatten()
    assert torch.equal(codes.flatten(), _nearest_even_bruteforce(flat))
    W = [O.expert_weight(inp, n, e) for n in ("w1", "w3", "w2")]
    o, a, a_codes = O.fp8_expert(codes, sx, sh, *W)
    assert torch.equal(a_codes.flatten(), _nearest_even_bruteforce(O.to_fp32(a * sh).flatten()))
    assert float((codes * O.dequant_multiplier(sx) - rows).abs().max()) <= \
        float(rows.abs().max()) * 2.0 ** -4 + 2.0 ** -10 / sx
    # the layer's own output for those tokens uses the same quantized rows
    toks = (out["idx"] == e).any(1).nonzero().flatten()
    j = (out["idx"][toks] == e).long().argmax(1)
    assert torch.allclose(out["o"][toks, j], o, rtol=1e-12, atol=1e-12)


def pin_mask_all_ones_is_no_mask():
    """An all-ones token mask changes nothing, bit for bit."""
    from moe_workloads import SHAPES, make_layer_inputs
    s = SHAPES["tiny_f32"].with_(T=48, capacity=(1, 2))
    inp = make_layer_inputs(s, "cpu")
    a = O.forward(inp, top_k=s.top_k, rms_eps=s.rms_eps, capacity_factor=s.capacity)
    inp1 = dict(inp, token_mask=torch.ones(s.T, dtype=torch.uint8))
    b = O.forward(inp1, top_k=s.top_k, rms_eps=s.rms_eps, capacity_factor=s.capacity)
    for key in ("counts", "offsets", "slot_of", "perm", "n_dropped", "y"):
        assert torch.equal(a[key], b[key]), key


def pin_mask_padding_keeps_shared_only():
    """Without capacity, a padding token's output is the shared path alone (the same layer with
    every routed W2 zero), and every other token's output is unchanged by the mask."""
    from moe_workloads import SHAPES, make_layer_inputs
    s = SHAPES["tiny_f32"].with_(T=40)
    inp = make_layer_inputs(s, "cpu")
    mask = torch.ones(s.T, dtype=torch.uint8)
    pad = [0, 7, 8, 39]
    mask[pad] = 0
    kw = dict(top_k=s.top_k, rms_eps=s.rms_eps)
    full = O.forward(inp, **kw)
    masked = O.forward(dict(inp, token_mask=mask), **kw)
    no_routed = O.forward(dict(inp, w2=torch.zeros_like(inp["w2"])), **kw)
    real = mask.bool()
    assert torch.allclose(masked["y"][~real], no_routed["y"][~real], rtol=0, atol=1e-14)
    assert torch.equal(masked["y"][real], full["y"][real])
    assert int(masked["counts"].sum()) == s.top_k * (s.T - len(pad))
    assert bool((masked["slot_of"][~real] == -1).all()) and int(masked["n_dropped"]) == 0


def pin_mask_frees_capacity():
    """Hand-derived: 4 tokens all choose expert 0 of 2 (k = 1) with capacity 2. Unmasked, tokens
    0 and 1 are kept and 2 and 3 dropped. With token 0 padding, tokens 1 and 2 take the two slots,
    token 3 is the only drop, and the padding token is neither counted nor dropped."""
    idx = torch.zeros((4, 1), dtype=torch.int64)
    d0 = O.dispatch(idx, 2, 2)
    assert d0["slot_of"].flatten().tolist() == [0, 1, -1, -1] and int(d0["n_dropped"]) == 2
    d = O.dispatch(idx, 2, 2, torch.tensor([0, 1, 1, 1]))
    assert d["counts"].tolist() == [3, 0]
    assert d["offsets"].tolist() == [0, 2, 2]
    assert d["slot_of"].flatten().tolist() == [-1, 0, 1, -1]
    assert d["perm"].tolist() == [1, 2]
    assert int(d["n_dropped"]) == 1


def _tiny_grouped(seed=5, E=3, L=6, F=5, counts=(3, 0, 4)):
    g = torch.Generator().manual_seed(seed)
    R = sum(counts)
    rows = torch.randn(R, L, generator=g, dtype=F64)
    w1 = torch.randn(E, L, F, generator=g, dtype=F64) * 0.5
    w3 = torch.randn(E, L, F, generator=g, dtype=F64) * 0.5
    w2 = torch.randn(E, F, L, generator=g, dtype=F64) * 0.5
    dy = torch.randn(R, L, generator=g, dtype=F64)
    offs = [0]
    for c in counts:
        offs.append(offs[-1] + c)
    return rows, offs, w1, w3, w2, dy


def pin_expert_backward_autograd():
    """The hand-written chain rule against torch.autograd of the SwiGLU expert definition
    y = (silu(x W1) * (x W3)) W2 per group: input and every weight gradient, an expert with no
    rows included. (The oracle's forward promotes without autograd; the finite-difference pin
    uses it as a black box.)"""
    rows, offs, w1, w3, w2, dy = _tiny_grouped()
    leaves = [t.clone().requires_grad_(True) for t in (rows, w1, w3, w2)]
    parts = []
    for e in range(len(offs) - 1):
        X = leaves[0][offs[e]:offs[e + 1]]
        parts.append((torch.nn.functional.silu(X @ leaves[1][e]) * (X @ leaves[2][e])) @ leaves[3][e])
    (torch.cat(parts) * dy).sum().backward()
    got = O.grouped_experts_backward(rows, offs, w1, w3, w2, dy)
    for name, leaf in zip(("dx", "dw1", "dw3", "dw2"), leaves):
        assert torch.allclose(got[name], leaf.grad, rtol=1e-12, atol=1e-12), name
    assert float(got["dw1"][1].abs().max()) == 0.0 and float(got["dw2"][1].abs().max()) == 0.0


def pin_expert_backward_finite_differences():
    """Central differences of <dy, y_perm> in fp64 for sampled entries of every gradient."""
    rows, offs, w1, w3, w2, dy = _tiny_grouped(seed=9, counts=(2, 5, 1))
    got = O.grouped_experts_backward(rows, offs, w1, w3, w2, dy)

    def loss(r, a, b, c):
        return float((O.grouped_experts(r, offs, a, b, c)[1] * dy).sum())
    h = 1e-6
    args = [rows, w1, w3, w2]
    for ai, name, index in ((0, "dx", (4, 2)), (1, "dw1", (1, 3, 2)), (2, "dw3", (2, 0, 4)),
                            (3, "dw2", (0, 1, 5)), (3, "dw2", (2, 4, 0))):
        plus = [t.clone() for t in args]
        minus = [t.clone() for t in args]
        plus[ai][index] += h
        minus[ai][index] -= h
        fd = (loss(*plus) - loss(*minus)) / (2 * h)
        assert abs(fd - float(got[name][index])) <= 1e-6 * (1 + abs(fd)), (name, fd)


def pin_silu_grad_closed_form():
    """silu'(0) = 1/2; silu'(v) -> 1 for large v and -> 0 for very negative v; against the
    derivative of v / (1 + e^-v) by central differences."""
    v = torch.tensor([0.0, 30.0, -40.0, 1.3, -2.7], dtype=F64)
    d = O.silu_grad(v)
    assert float(d[0]) == 0.5
    assert abs(float(d[1]) - 1.0) < 1e-11 and abs(float(d[2])) < 1e-15
    h = 1e-6
    fd = (O.silu(v[3:] + h) - O.silu(v[3:] - h)) / (2 * h)
    assert torch.allclose(d[3:], fd, rtol=0, atol=1e-9)


def _tiny_layer(seed=13, cap=None):
    """A random fp64 layer small enough for finite differences over every weight."""
    g = torch.Generator().manual_seed(seed)
    T, d, L, E, k, F, S, Fs = 6, 8, 6, 4, 2, 5, 1, 4
    r = lambda *sh: torch.randn(*sh, generator=g, dtype=F64)
    inp = {"x": r(T, d), "w_router": r(d, E), "b_router": r(E) * 0.3, "w_down": r(d, L) * 0.4,
           "rms_gamma": 1.0 + 0.2 * r(L), "w1": r(E, L, F) * 0.5, "w3": r(E, L, F) * 0.5,
           "w2": r(E, F, L) * 0.5, "w1_s": r(S, d, Fs) * 0.4, "w3_s": r(S, d, Fs) * 0.4,
           "w2_s": r(S, Fs, d) * 0.4, "w_up": r(L, d) * 0.4}
    return inp, r(T, d), dict(top_k=k, rms_eps=1e-6, capacity_factor=cap)


def pin_layer_backward_finite_differences():
    """Central differences of <dy, y> through the oracle's forward, for sampled entries of every
    gradient, with and without a capacity that drops assignments (routing is unchanged by the
    1e-6 perturbations of these random inputs)."""
    for cap in (None, (1, 2)):
        inp, dy, kw = _tiny_layer(cap=cap)
        fwd = O.forward(inp, **kw)
        if cap:
            assert int(fwd["n_dropped"]) > 0
        got = O.backward(inp, fwd, dy, rms_eps=kw["rms_eps"])

        def loss(mod):
            return float((O.forward(mod, **kw)["y"] * dy).sum())
        h = 1e-6
        checks = [("x", "dx", (2, 3)), ("x", "dx", (5, 0)), ("w_router", "dw_router", (1, 2)),
                  ("w_router", "dw_router", (7, 0)), ("b_router", "db_router", (3,)),
                  ("w_down", "dw_down", (4, 1)), ("rms_gamma", "drms_gamma", (2,)),
                  ("w1", "dw1", (int(fwd["idx"][0, 0]), 1, 2)),
                  ("w3", "dw3", (int(fwd["idx"][1, 1]), 0, 4)),
                  ("w2", "dw2", (int(fwd["idx"][2, 0]), 3, 5)),
                  ("w1_s", "dw1_s", (0, 6, 1)), ("w3_s", "dw3_s", (0, 2, 3)),
                  ("w2_s", "dw2_s", (0, 1, 7)), ("w_up", "dw_up", (5, 6))]
        for wname, gname, index in checks:
            plus, minus = dict(inp), dict(inp)
            plus[wname] = inp[wname].clone()
            minus[wname] = inp[wname].clone()
            plus[wname][index] += h
            minus[wname][index] -= h
            fd = (loss(plus) - loss(minus)) / (2 * h)
            an = float(got[gname][index])
            assert abs(fd - an) <= 1e-6 * (1 + abs(fd)), (cap, gname, index, fd, an)


def pin_layer_backward_dx_without_expert_weight_grads():
    """Leaving out the routed experts' weight gradients (for a dx check on a bank too large for
    fp64 copies) changes no other output: every remaining gradient is identical."""
    inp, dy, kw = _tiny_layer(cap=None)
    fwd = O.forward(inp, **kw)
    full = O.backward(inp, fwd, dy, rms_eps=kw["rms_eps"])
    part = O.backward(inp, fwd, dy, rms_eps=kw["rms_eps"], expert_weight_grads=False)
    assert set(full) - set(part) == {"dw1", "dw3", "dw2"}
    for n in part:
        assert torch.equal(part[n], full[n]), n


ALL_PINS = [pin_layer_backward_dx_without_expert_weight_grads, pin_layer_backward_finite_differences, pin_expert_backward_autograd, pin_expert_backward_finite_differences,
            pin_silu_grad_closed_form, pin_mask_all_ones_is_no_mask, pin_mask_padding_keeps_shared_only,
            pin_mask_frees_capacity, pin_fp8_expert_golden, pin_e4m3_rounding, pin_fp8_quantize_in_fp32,
            pin_fp8_layer_grid, pin_forward_drop_skips_expert, pin_topk_bruteforce, pin_topk_exact_near_tie, pin_logit_bound_holds, pin_gates,
            pin_capacity, pin_dispatch_golden, pin_dispatch_invariants, pin_forced_single_expert,
            pin_identical_experts, pin_two_token_golden, pin_rmsnorm,
            pin_combine_drop_not_renormalised, pin_slice_rowwise]


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(pin):
    pin()


# -------------------------------------------------------- planted mistakes ----

def _mut_silu_no_sigmoid(monkeypatch):
    monkeypatch.setattr(O, "silu", lambda v: v * torch.exp(-v))


def _mut_tie_high_index(monkeypatch):
    orig = O.topk_exact

    def bad(logits, bound, k, exact_fn):
        E = logits.shape[1]
        flipped = orig(logits.flip(1), bound.flip(1), k, lambda t, e: exact_fn(t, E - 1 - e))
        return torch.sort(E - 1 - flipped, dim=1).values
    monkeypatch.setattr(O, "topk_exact", bad)


def _mut_float_capacity(monkeypatch):
    monkeypatch.setattr(O, "capacity", lambda T, k, E, cf: None if cf is None or cf[0] <= 0
                        else math.ceil(cf[0] / cf[1] * T * k / E))


def _mut_no_shared(monkeypatch):
    monkeypatch.setattr(O, "shared_hidden", lambda x, w1, w3: torch.zeros(
        x.shape[0], w1.shape[0] * w1.shape[2], dtype=F64))


def _mut_rms_sum(monkeypatch):
    def bad(x, w_down, gamma, eps):
        z = O.to64(x) @ O.to64(w_down)
        return z, z / torch.sqrt((z * z).sum(1, keepdim=True) + eps) * O.to64(gamma)
    monkeypatch.setattr(O, "latent", bad)


def _mut_full_softmax(monkeypatch):
    monkeypatch.setattr(O, "softmax_gates",
                        lambda logits, idx: torch.softmax(logits, 1).gather(1, idx))


def _mut_renorm_after_drop(monkeypatch):
    orig = O.combine

    def bad(y_perm, slot_of, gate):
        g = gate.clone().double() * (slot_of >= 0)
        g = g / g.sum(1, keepdim=True).clamp_min(1e-300)
        return orig(y_perm, slot_of, g)
    monkeypatch.setattr(O, "combine", bad)


def _mut_forward_renorm(monkeypatch):
    orig = O.softmax_gates

    def bad(logits, idx):                   # gates computed as if dropped experts never existed
        g = orig(logits, idx)
        return g * 0.5 + 0.5 / idx.shape[1]
    monkeypatch.setattr(O, "softmax_gates", bad)


def _mut_fp8_scale_ignored(monkeypatch):
    monkeypatch.setattr(O, "expert_weight", lambda inp, name, e: O.to64(inp[name][e]))


def _mut_e4m3_ties_away(monkeypatch):
    def bad(v):
        v = O.to64(v)
        a = v.abs()
        _, ex = torch.frexp(a)
        step = torch.exp2((torch.clamp(ex - 1, min=-6) - 3).to(F64))
        return torch.sign(v) * torch.clamp(torch.floor(a / step + 0.5) * step, max=448.0)
    monkeypatch.setattr(O, "e4m3_round", bad)


def _mut_fp8_no_activation_rounding(monkeypatch):
    monkeypatch.setattr(O, "quantize_e4m3", lambda v, scale: O.to64(v) * float(scale))


def _mut_fp8_dequant_by_scale(monkeypatch):
    monkeypatch.setattr(O, "dequant_multiplier", lambda scale: float(scale))


def _mut_fp8_quantize_in_fp64(monkeypatch):
    monkeypatch.setattr(O, "quantize_e4m3", lambda v, scale: O.e4m3_round(O.to64(v) * float(scale)))


def _mut_mask_ignored(monkeypatch):
    orig = O.dispatch
    monkeypatch.setattr(O, "dispatch", lambda idx, E, cap, mask=None: orig(idx, E, cap))


def _mut_mask_counts_padding(monkeypatch):
    orig = O.dispatch

    def bad(idx, E, cap, mask=None):
        d = orig(idx, E, cap, mask)
        if mask is not None:   # padding assignments still counted before the clamp
            full = orig(idx, E, cap)
            d["counts"] = full["counts"]
        return d
    monkeypatch.setattr(O, "dispatch", bad)


def _mut_silu_grad_no_inner(monkeypatch):
    monkeypatch.setattr(O, "silu_grad", lambda v: 1.0 / (1.0 + torch.exp(-v)))


def _mut_backward_dw2_from_g(monkeypatch):
    orig = O.grouped_experts_backward

    def bad(rows, offsets, w1, w3, w2, dy, **kw):
        out = orig(rows, offsets, w1, w3, w2, dy, **kw)
        for e in range(len(offsets) - 1):
            lo, hi = int(offsets[e]), int(offsets[e + 1])
            if hi > lo and "dw2" in out:
                out["dw2"][e] = out["g"][lo:hi].T @ O.to64(dy)[lo:hi]
        return out
    monkeypatch.setattr(O, "grouped_experts_backward", bad)


def _mut_backward_dx_no_w3(monkeypatch):
    orig = O.grouped_experts_backward

    def bad(rows, offsets, w1, w3, w2, dy, **kw):
        out = orig(rows, offsets, w1, w3, w2, dy, **kw)
        for e in range(len(offsets) - 1):
            lo, hi = int(offsets[e]), int(offsets[e + 1])
            if hi > lo:
                out["dx"][lo:hi] = out["dg"][lo:hi] @ O.to64(w1[e]).T
        return out
    monkeypatch.setattr(O, "grouped_experts_backward", bad)


def _mut_router_grad_full_softmax(monkeypatch):
    orig = O.backward

    def bad(inp, fwd, dy, *, rms_eps, **kw):
        out = orig(inp, fwd, dy, rms_eps=rms_eps, **kw)
        # forget the normalisation over the selected experts: dl_j = g_j dg_j
        dl = torch.zeros((fwd["idx"].shape[0], inp["w_router"].shape[1]), dtype=F64)
        for j in range(fwd["idx"].shape[1]):
            dl[torch.arange(dl.shape[0]), fwd["idx"][:, j]] += fwd["gate"][:, j] * out["dgate"][:, j]
        out["dw_router"] = O.to64(inp["x"]).T @ dl
        return out
    monkeypatch.setattr(O, "backward", bad)


def _mut_rmsnorm_grad_no_projection(monkeypatch):
    orig = O.backward

    def bad(inp, fwd, dy, *, rms_eps, **kw):
        out = orig(inp, fwd, dy, rms_eps=rms_eps, **kw)
        z = fwd["z"]
        rstd = 1.0 / torch.sqrt((z * z).mean(dim=1, keepdim=True) + rms_eps)
        dz = rstd * out["dh"] * O.to64(inp["rms_gamma"])         # drops the mean term
        out["dw_down"] = O.to64(inp["x"]).T @ dz
        return out
    monkeypatch.setattr(O, "backward", bad)


def _mut_unstable_perm(monkeypatch):
    orig = O.dispatch

    def bad(idx, E, cap, mask=None):
        d = orig(idx.flip(0), E, cap, None if mask is None else mask.flip(0))   # reverse order
        d["slot_of"] = d["slot_of"].flip(0)
        T, k = idx.shape
        d["perm"] = torch.where(d["perm"] >= 0, (T - 1 - d["perm"] // k) * k + d["perm"] % k,
                                d["perm"])
        return d
    monkeypatch.setattr(O, "dispatch", bad)


def _mut_slice_rows_boundary(monkeypatch):
    """slice_rows assigns a pool row to the first group whose end is >= the row (an off-by-one
    at a group boundary)."""
    def bad(inp, positions):
        offs = [int(v) for v in inp["expert_offsets"].tolist()]
        pos = [int(p) for p in positions]
        rows = [int(inp["slot_of"][p]) for p in pos]
        o = torch.zeros((len(pos), inp["w2"].shape[2]), dtype=F64)
        for n, r in enumerate(rows):
            e = min(g for g in range(len(offs) - 1) if offs[g + 1] >= r)
            v = O.to64(inp["pool"][[r]])
            o[n] = O.swiglu_mlp(v, O.expert_weight(inp, "w1", e), O.expert_weight(inp, "w3", e),
                                O.expert_weight(inp, "w2", e))[0]
        g = O.to64(inp["gate"][pos]).unsqueeze(1)
        return {"rows": torch.tensor(rows), "y_perm": o, "out": g * o}
    monkeypatch.setattr(O, "slice_rows", bad)


def _mut_slice_rows_gate_by_row(monkeypatch):
    """slice_rows weights by the gate of the pool row instead of the arrival position."""
    orig = O.slice_rows

    def bad(inp, positions):
        res = orig(inp, positions)
        g_row = O.to64(inp["gate"][res["rows"].clamp(max=inp["gate"].numel() - 1)]).unsqueeze(1)
        return {**res, "out": g_row * res["y_perm"]}
    monkeypatch.setattr(O, "slice_rows", bad)


def _mut_transposed_up(monkeypatch):
    orig = O.forward

    def bad(inp, **kw):
        inp = dict(inp)
        L, d = inp["w_up"].shape
        inp["w_up"] = inp["w_up"].t().reshape(L, d) if L != d else inp["w_up"].t()
        return orig(inp, **kw)
    monkeypatch.setattr(O, "forward", bad)


MUTATIONS = [_mut_silu_no_sigmoid, _mut_tie_high_index, _mut_float_capacity, _mut_no_shared,
             _mut_rms_sum, _mut_full_softmax, _mut_renorm_after_drop, _mut_forward_renorm, _mut_fp8_scale_ignored, _mut_e4m3_ties_away,
             _mut_fp8_no_activation_rounding, _mut_fp8_dequant_by_scale,
             _mut_fp8_quantize_in_fp64, _mut_mask_ignored, _mut_mask_counts_padding,
             _mut_silu_grad_no_inner, _mut_backward_dw2_from_g, _mut_backward_dx_no_w3,
             _mut_router_grad_full_softmax, _mut_rmsnorm_grad_no_projection,
             _mut_unstable_perm,
             _mut_transposed_up, _mut_slice_rows_boundary, _mut_slice_rows_gate_by_row]


@pytest.mark.parametrize("mutate", MUTATIONS, ids=[m.__name__[5:] for m in MUTATIONS])
def test_planted_mistakes_are_caught(mutate, monkeypatch):
    mutate(monkeypatch)
    caught = []
    for pin in ALL_PINS:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {mutate.__name__}"
