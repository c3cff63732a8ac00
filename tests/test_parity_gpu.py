"""Parity of the CUDA library (through its C ABI) with the fp64 oracle on seeded inputs.

Bar: routing indices, expert counts, offsets, slots and drops bit-exact; gates within 1e-6
(fp32 configuration) / 1e-5 (bf16); outputs within a normwise relative error of 1e-5 (fp32)
and 2e-2 (bf16 storage of the intermediates, fp32 accumulation).
"""
import pytest
import torch

import sparse_expert_router_gb300 as m
from moe_workloads import SHAPES, SLICE_C5B, make_layer_inputs, make_slice_inputs, padding_mask
from oracle import moe_oracle

from gpu_cases import (DEV, check_routing, e4m3_codes_match, gpu_inputs, near_tie_router, normwise,
                       oracle_forward, run_forward, sample_tokens)

pytestmark = pytest.mark.gpu

# the bf16 GEMM paths under test: tensor cores (default), tensor cores with programmatic
# dependent launch (the bench configuration) and the CUDA-core cross-check
BF16_PATHS = {"tc": 0, "tc_pdl": m.MOE_FLAG_PDL, "simt": m.MOE_FLAG_SIMT}
def _check_combine(shape, cfg, got):
    """The combine c the forward left in its workspace (computed inside the back GEMM's launch
    for tensor-core layers with shared experts) against the separate combine kernel on the same
    y_perm, slots and gates (moe_combine without an up-projection), bit for bit, and against the
    oracle's combine of those rows in fp64 (bf16 rounding of c: at most 2^-8 per element)."""
    T, L = shape.T, shape.d_latent
    P = T * shape.top_k
    ws = got["ws"]
    c = m.workspace_view(ws, cfg, "combined", torch.bfloat16, (T, L)).clone()
    yp = m.workspace_view(ws, cfg, "y_perm", torch.bfloat16, (P, L))
    gate = got["topk_gate"]
    sep = torch.empty((T, L), dtype=torch.bfloat16, device=DEV)
    m.moe_combine(cfg, yp, got["slot_of"], gate, sep, ws)
    torch.cuda.synchronize()
    assert torch.equal(c.view(torch.int16), sep.view(torch.int16))
    toks = sample_tokens(T, 64)
    slots = got["slot_of"].cpu().long()[toks]                  # [64, k], -1 = dropped
    rows = yp[slots.clamp(min=0).flatten().to(DEV)]            # the rows those slots name
    local = torch.where(slots >= 0, torch.arange(slots.numel()).view(slots.shape), -1)
    ref = moe_oracle.combine(rows, local, gate.cpu()[toks])
    err = (c[toks].double().cpu() - ref).abs() - 2.0 ** -8 * ref.abs()
    assert float(err.max()) <= 1e-6, float(err.max())


# The bench configuration runs with programmatic dependent launch on (MOE_FLAG_PDL); the
# full-size and edge-case forwards run both with and without it.
PDL_FLAGS = {"nopdl": 0, "pdl": m.MOE_FLAG_PDL}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


# ------------------------------------------------------------------ full layer, small ----

@pytest.mark.parametrize("flags", [0, m.MOE_FLAG_PDL], ids=["nopdl", "pdl"])
@pytest.mark.parametrize("cap", [None, (11, 10), (1, 2)], ids=["nocap", "cf110", "cf050"])
def test_tiny_f32_forward(cap, flags):
    shape = SHAPES["tiny_f32"].with_(capacity=cap)
    inp = gpu_inputs(shape)
    got = run_forward(shape, inp, flags)
    ref = oracle_forward(shape, {k: v.cpu() for k, v in inp.items()})
    check_routing(got, ref, shape)
    if cap == (1, 2):
        assert int(ref["n_dropped"]) > 0
    err = normwise(got["y"], ref["y"])
    assert err <= 1e-5, err
    assert got["report"]["status"] == 0


@pytest.mark.parametrize("path", list(BF16_PATHS))
def test_small_bf16_forward(path):
    shape = SHAPES["small_bf16"]
    inp = gpu_inputs(shape)
    got = run_forward(shape, inp, BF16_PATHS[path])
    if path != "simt":
        _check_combine(shape, m.LayerConfig.from_shape(shape, flags=BF16_PATHS[path]), got)
    toks = sample_tokens(shape.T, 256)
    ref = oracle_forward(shape, {k: v.cpu() for k, v in inp.items()}, tokens=toks)
    check_routing(got, ref, shape)
    err = normwise(got["y"][toks], ref["y"])
    assert err <= 2e-2, err
    assert got["report"]["status"] == 0


def test_forward_deterministic():
    """Two runs give the same bits: bf16 on both GEMM paths, and fp8 experts (whose amax
    reductions are order-independent maxima)."""
    shape = SHAPES["small_bf16"].with_(T=1024)
    inp = gpu_inputs(shape)
    for flags in BF16_PATHS.values():
        a = run_forward(shape, inp, flags)
        b = run_forward(shape, inp, flags)
        assert torch.equal(a["y"].view(torch.int16), b["y"].view(torch.int16))
        assert torch.equal(a["topk_gate"], b["topk_gate"])
    shape = SHAPES["small_fp8"].with_(T=1024)
    inp = gpu_inputs(shape)
    a, b = run_forward(shape, inp), run_forward(shape, inp)
    assert torch.equal(a["y"].view(torch.int16), b["y"].view(torch.int16))
    assert float(a["x_amax"]) == float(b["x_amax"]) and float(a["h_amax"]) == float(b["h_amax"])


# ---------------------------------------------------------------------- split calls ----

def test_split_calls_tiny_f32():
    shape = SHAPES["tiny_f32"].with_(capacity=(1, 2))
    cfg = m.LayerConfig.from_shape(shape)
    cpu = make_layer_inputs(shape, "cpu")
    inp = {k: v.to(DEV) for k, v in cpu.items()}
    T, k, E, L, F = shape.T, shape.top_k, shape.n_experts, shape.d_latent, shape.d_ff
    ws = m.alloc_workspace(cfg, DEV)
    ref = oracle_forward(shape, cpu)

    # moe_route
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, k), dtype=torch.float32, device=DEV)
    m.moe_route(cfg, inp["x"], inp["w_router"], inp["b_router"], idx, gate, ws)
    assert torch.equal(idx.cpu().long(), ref["idx"])
    assert float((gate.cpu().double() - ref["gate"]).abs().max()) <= 1e-6

    # moe_permute on the oracle's routing
    oidx = ref["idx"].to(torch.int32).to(DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.full((T * k,), -5, dtype=torch.int32, device=DEV)
    slot = torch.empty((T, k), dtype=torch.int32, device=DEV)
    ndrop = torch.empty(1, dtype=torch.int32, device=DEV)
    x_perm = torch.zeros((T * k, L), dtype=torch.float32, device=DEV)
    m.moe_permute(cfg, inp["x"], inp["w_down"], inp["rms_gamma"], oidx, counts, offs, perm, slot,
                  ndrop, x_perm, ws)
    assert torch.equal(counts.cpu().long(), ref["counts"])
    assert torch.equal(offs.cpu().long(), ref["offsets"])
    assert torch.equal(slot.cpu().long(), ref["slot_of"])
    R = int(ref["offsets"][-1])
    assert torch.equal(perm.cpu().long()[:R], ref["perm"])
    assert int(ndrop.cpu()) == int(ref["n_dropped"])
    # rows of x_perm are the normalised latent of their token
    tok = ref["perm"] // k
    assert normwise(x_perm[:R], ref["h"][tok]) <= 1e-5

    # moe_expert_ffn on the oracle's grouped rows (rounded to the storage type)
    xp = ref["h"][tok].float().to(DEV)
    y_perm = torch.zeros((T * k, L), dtype=torch.float32, device=DEV)
    a_s = torch.empty((T, shape.n_shared * shape.d_ff_shared), dtype=torch.float32, device=DEV)
    offs_in = ref["offsets"].to(torch.int32).to(DEV)
    xp_full = torch.zeros((T * k, L), dtype=torch.float32, device=DEV)
    xp_full[:R] = xp
    m.moe_expert_ffn(cfg, xp_full, offs_in, inp["w1"], inp["w3"], inp["w2"], y_perm, inp["x"],
                     inp["w1_s"], inp["w3_s"], a_s, ws)
    _, o_ref = moe_oracle.grouped_experts(xp_full.cpu(), ref["offsets"].tolist(), cpu["w1"],
                                          cpu["w3"], cpu["w2"])
    assert normwise(y_perm[:R], o_ref) <= 1e-5
    assert float(y_perm[R:].abs().max()) == 0.0          # rows past the groups untouched
    assert normwise(a_s, ref["a_s"]) <= 1e-5

    # moe_combine without and with the up-projection
    yp_in = o_ref.float().to(DEV)
    yp_full = torch.zeros((T * k, L), dtype=torch.float32, device=DEV)
    yp_full[:R] = yp_in
    c = torch.empty((T, L), dtype=torch.float32, device=DEV)
    ogate = ref["gate"].float().to(DEV)
    oslot = ref["slot_of"].to(torch.int32).to(DEV)
    m.moe_combine(cfg, yp_full, oslot, ogate, c, ws)
    c_ref = moe_oracle.combine(yp_full.cpu(), ref["slot_of"], ogate.cpu())
    assert normwise(c, c_ref) <= 1e-6
    y = torch.empty((T, shape.d_model), dtype=torch.float32, device=DEV)
    m.moe_combine(cfg, yp_full, oslot, ogate, y, ws, a_shared=ref["a_s"].float().to(DEV),
                  w_up=inp["w_up"], w2_s=inp["w2_s"])
    y_ref = c_ref @ cpu["w_up"].double() + ref["a_s"] @ cpu["w2_s"].double().reshape(-1, shape.d_model)
    assert normwise(y, y_ref) <= 1e-5
    assert m.moe_get_device_status(ws)["status"] == 0


# ----------------------------------------------------------- router exactness stress ----

@pytest.mark.parametrize("T", [48, 512])
@pytest.mark.parametrize("path", list(BF16_PATHS))
def test_router_exact_on_near_ties(path, T):
    """Nearly every token reaches the exact stage. The library keeps the stage-2 state of the
    first 64 of them and splits their exact stage over several blocks; the rest recompute
    stage 2 on one block each: T=48 takes only the first way, T=512 both."""
    x, w = near_tie_router(T=T)
    T, d = x.shape
    E, k = w.shape[1], 8
    cfg = m.LayerConfig(T=T, d_model=d, d_latent=64, n_experts=E, top_k=k, d_ff=64, n_shared=0,
                        d_ff_shared=0, dtype="bf16", flags=BF16_PATHS[path])
    ws = m.alloc_workspace(cfg, DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, k), dtype=torch.float32, device=DEV)
    m.moe_route(cfg, x.to(DEV), w.to(DEV), None, idx, gate, ws)
    rep = m.moe_get_device_status(ws)
    ref = moe_oracle.route(x, w, None, k)
    assert torch.equal(idx.cpu().long(), ref["idx"])
    assert rep["status"] == 0
    assert rep["n_refined"] > 0 and rep["n_exact"] > 0, rep      # every stage exercised
    if T > 64:
        assert rep["n_exact"] > 64, rep                           # past the saved slots too


@pytest.mark.parametrize("E,k,dtype,path", [(64, 8, "bf16", "tc"), (64, 8, "bf16", "simt"),
                                             (64, 8, "f32", "tc"), (1024, 32, "bf16", "tc")],
                         ids=["e64_bf16_tc", "e64_bf16_simt", "e64_f32", "e1024_k32_bf16"])
def test_router_tied_logits(E, k, dtype, path):
    """The degenerate router: zero weights, so every logit is its bias, and the biases repeat
    in four levels. The top level holds E/4 exactly equal logits; the k lowest indices among
    them win, and the gates are all 1/k. Every expert of the top level is undecided until the
    exact stage."""
    T, d = 40, 256
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator().manual_seed(5)
    x = torch.randn(T, d, generator=g).to(tdt)
    w = torch.zeros(d, E, dtype=tdt)
    b = (torch.arange(E) % 4).float() * 0.5
    cfg = m.LayerConfig(T=T, d_model=d, d_latent=64, n_experts=E, top_k=k, d_ff=64, n_shared=0,
                        d_ff_shared=0, dtype=dtype, flags=BF16_PATHS[path])
    ws = m.alloc_workspace(cfg, DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, k), dtype=torch.float32, device=DEV)
    m.moe_route(cfg, x.to(DEV), w.to(DEV), b.to(DEV), idx, gate, ws)
    rep = m.moe_get_device_status(ws)
    ref = moe_oracle.route(x, w, b, k)
    want = torch.arange(3, 4 * k, 4).expand(T, -1)
    assert torch.equal(ref["idx"], want)                          # the oracle's own reading
    assert torch.equal(idx.cpu().long(), want)
    assert float((gate.cpu() - 1.0 / k).abs().max()) <= 1e-7
    assert rep["status"] == 0
    assert rep["n_exact"] == T, rep


def test_router_exact_on_near_ties_f32():
    """The same near ties with fp32 router inputs: stage 2 then needs TwoProduct for the exact
    products of fp32 values, and stage 3 integer products of 24-bit significands."""
    x, w = near_tie_router(T=512, dtype=torch.float32)
    T, d = x.shape
    E, k = w.shape[1], 8
    cfg = m.LayerConfig(T=T, d_model=d, d_latent=64, n_experts=E, top_k=k, d_ff=64, n_shared=0,
                        d_ff_shared=0, dtype="f32")
    ws = m.alloc_workspace(cfg, DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, k), dtype=torch.float32, device=DEV)
    m.moe_route(cfg, x.to(DEV), w.to(DEV), None, idx, gate, ws)
    rep = m.moe_get_device_status(ws)
    ref = moe_oracle.route(x, w, None, k)
    assert torch.equal(idx.cpu().long(), ref["idx"])
    assert float((gate.cpu().double() - ref["gate"]).abs().max()) <= 1e-6
    assert rep["status"] == 0
    assert rep["n_refined"] > 0 and rep["n_exact"] > 64, rep      # both exact-stage paths


# ------------------------------------------------------------ device-detected errors ----

def test_bad_routing_is_reported_not_faulted():
    shape = SHAPES["tiny_f32"]
    cfg = m.LayerConfig.from_shape(shape)
    cpu = make_layer_inputs(shape, "cpu")
    inp = {k: v.to(DEV) for k, v in cpu.items()}
    T, k, E, L = shape.T, shape.top_k, shape.n_experts, shape.d_latent
    ws = m.alloc_workspace(cfg, DEV)
    bad = torch.stack([torch.arange(k) for _ in range(T)]).to(torch.int32)
    bad[5, 1] = E + 3                                # out of range
    bad[9] = torch.tensor([4, 4])                    # repeated expert
    bad = bad.to(DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    slot = torch.empty((T, k), dtype=torch.int32, device=DEV)
    x_perm = torch.zeros((T * k, L), dtype=torch.float32, device=DEV)
    m.moe_clear_device_status(ws)
    m.moe_permute(cfg, inp["x"], inp["w_down"], inp["rms_gamma"], bad, counts, offs, perm, slot,
                  None, x_perm, ws)
    rep = m.moe_get_device_status(ws)
    assert rep["status"] == 6, rep                   # MOE_ERR_BAD_ROUTING
    assert int(slot[5, 1]) == -1 and int(slot[9, 1]) == -1
    assert int(counts.sum()) == T * k - 2

    # non-monotone offsets into the grouped GEMM: reported, and nothing out of range runs
    m.moe_clear_device_status(ws)
    offs_bad = torch.tensor([0, 40, 20, 10**6] + [10**6] * (E - 3), dtype=torch.int32, device=DEV)
    y_perm = torch.zeros((T * k, L), dtype=torch.float32, device=DEV)
    m.moe_expert_ffn(cfg, x_perm, offs_bad, inp["w1"], inp["w3"], inp["w2"], y_perm, ws=ws)
    rep = m.moe_get_device_status(ws)
    assert rep["status"] == 6, rep
    torch.cuda.synchronize()


def test_bounded_wait_times_out_and_context_survives():
    """Failure detection without a fault: a bounded device wait that nothing satisfies gives up
    after its limit, the host reads MOE_ERR_DEVICE_TIMEOUT, and the GPU keeps working."""
    import time
    shape = SHAPES["tiny_f32"]
    cfg = m.LayerConfig.from_shape(shape)
    ws = m.alloc_workspace(cfg, DEV)
    t0 = time.perf_counter()
    m.moe_selftest_device_timeout(ws, 200)
    rep = m.moe_get_device_status(ws)
    dt = time.perf_counter() - t0
    assert rep["status"] == 7 and rep["detail"] == 99, rep      # MOE_ERR_DEVICE_TIMEOUT
    assert 0.15 < dt < 5.0, dt
    # the context is intact: a forward right after runs and matches the oracle's routing
    inp = gpu_inputs(shape)
    got = run_forward(shape, inp)
    ref = oracle_forward(shape, {k: v.cpu() for k, v in inp.items()})
    check_routing(got, ref, shape)
    assert got["report"]["status"] == 0


# ------------------------------------------------------------------- 535B-shaped ----

LARGE = ["l535b_t8192", "l535b_zipf_t16384", "l535b_zipf_t16384_cf110", "l535b_t65536",
         "l535b_t8192_fp8"]


def _chosen_experts(offs):
    """The three experts with the most grouped rows, the one with the fewest (non-empty) and the
    one in the middle of the non-empty experts ordered by rows."""
    rows = offs[1:] - offs[:-1]
    nz = (rows > 0).nonzero().flatten()
    order = nz[rows[nz].argsort(stable=True)]
    picks = [int(order[-1]), int(order[-2]), int(order[-3]), int(order[0]),
             int(order[len(order) // 2])]
    return list(dict.fromkeys(picks))


def _check_expert_rows(shape, inp, cfg, ws, offs, name):
    """Every grouped row of the chosen experts, read from the forward's workspace: the rows the
    gather wrote (x_perm) against the oracle's normalised latent of their tokens, the SwiGLU
    hidden and the expert outputs (y_perm) against the oracle's expert MLP on those same rows.
    Per-expert and per-row normwise bounds."""
    P, L, F, k = shape.T * shape.top_k, shape.d_latent, shape.d_ff, shape.top_k
    fp8 = shape.expert_dtype == "fp8"
    xdt = torch.uint8 if fp8 else torch.bfloat16
    xp = m.workspace_view(ws, cfg, "x_perm", xdt, (P, L))
    hid = m.workspace_view(ws, cfg, "hidden", xdt, (P, F))
    yp = m.workspace_view(ws, cfg, "y_perm", torch.bfloat16, (P, L))
    perm = m.workspace_view(ws, cfg, "perm", torch.int32, (P,))
    scales = {n: inp[n] for n in ("w1_scale", "w3_scale", "w2_scale", "x_scale", "h_scale")} \
        if fp8 else None
    checked = 0
    for e in _chosen_experts(offs):
        lo, hi = int(offs[e]), int(offs[e + 1])
        tok = (perm[lo:hi].long() // k).cpu()
        if fp8:
            rows = xp[lo:hi].view(torch.float8_e4m3fn).to(torch.float64).cpu()
        else:
            rows = xp[lo:hi]
            _, h = moe_oracle.latent(inp["x"][tok.to(DEV)], inp["w_down"], inp["rms_gamma"],
                                     shape.rms_eps)
            r64 = rows.double().cpu()
            err_h = (r64 - h).norm(dim=1) / h.norm(dim=1).clamp_min(1e-300)
            assert float(err_h.max()) <= 4e-3, (name, e, "x_perm", float(err_h.max()))
        a, o = moe_oracle.grouped_experts(
            rows, [0, hi - lo], inp["w1"][e:e + 1], inp["w3"][e:e + 1], inp["w2"][e:e + 1],
            fp8={**scales, **{n: scales[n][e:e + 1] for n in ("w1_scale", "w3_scale", "w2_scale")}}
            if fp8 else None)
        got = yp[lo:hi].double().cpu()
        assert normwise(got, o) <= 2e-2, (name, e, hi - lo)
        per_row = ((got - o).norm(dim=1) / o.norm(dim=1).clamp_min(1e-300))
        assert float(per_row.max()) <= 2e-2, (name, e, hi - lo, float(per_row.max()))
        if not fp8:
            assert normwise(hid[lo:hi], a) <= 2e-2, (name, e, "hidden")
        checked += hi - lo
    return checked


@pytest.mark.parametrize("name", LARGE)
def test_large_layer(name):
    """Full routing and dispatch checked bit-exactly on every token, with and without PDL, and the
    two outputs bitwise equal. Outputs of 256 seeded tokens plus the hottest expert's first tokens
    and dropped tokens against the oracle (each token's output depends only on its own row and
    routing), normwise over the sample and per token. Every grouped row of five experts (the
    three hottest, the smallest and a middle one) read from the PDL forward's workspace: gathered
    rows, hidden and expert outputs against the oracle."""
    shape = SHAPES[name]
    inp = gpu_inputs(shape)
    runs = {f: run_forward(shape, inp, PDL_FLAGS[f]) for f in PDL_FLAGS}
    got = runs["pdl"]
    assert torch.equal(runs["pdl"]["y"].view(torch.int16), runs["nopdl"]["y"].view(torch.int16))
    counts = got["expert_counts"].cpu()
    hot = int(counts.argmax())
    hot_tokens = (got["topk_idx"].cpu() == hot).any(1).nonzero().flatten()[:4].tolist()
    dropped = (got["slot_of"].cpu() < 0).any(1).nonzero().flatten()[:4].tolist()
    toks = sample_tokens(shape.T, 256, extra=hot_tokens + dropped)
    ref = oracle_forward(shape, inp, tokens=toks)
    for f in PDL_FLAGS:
        check_routing(runs[f], ref, shape)
        assert runs[f]["report"]["status"] == 0
    if shape.routing == "zipf":
        assert int((counts == 0).sum()) > 0                      # experts with no rows
        assert float(counts.max()) > 20 * shape.T * shape.top_k / shape.n_experts
    if shape.capacity:
        assert int(ref["n_dropped"]) > 0
    ys = got["y"][toks].double().cpu()
    assert normwise(ys, ref["y"]) <= 2e-2
    per_tok = (ys - ref["y"]).norm(dim=1) / ref["y"].norm(dim=1).clamp_min(1e-300)
    assert float(per_tok.max()) <= 2e-2, float(per_tok.max())
    cfg = m.LayerConfig.from_shape(shape, flags=PDL_FLAGS["pdl"])
    n_rows = _check_expert_rows(shape, inp, cfg, got["ws"], got["expert_offsets"].cpu(), name)
    assert n_rows > 0
    _check_combine(shape, cfg, got)
    del inp, got, runs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("path", ["tc", "tc_pdl", "f32"])
def test_swiglu_epilogue_wide_range(path):
    """The grouped GEMM's SwiGLU epilogue on its own, over gate pre-activations u1 in [-30, 30] and
    up pre-activations u3 in [-4, 4]: one-hot rows (row r is e_{r mod L}) make u1 = W1[r mod L, f]
    and u3 = W3[r mod L, f] exactly, so the stored hidden silu(u1) * u3 is compared element by
    element with the oracle's fp64 value. Bar: the rounding to the stored type (bf16, with its
    8-bit significand: at most 2^-8 relative) plus 2e-5 relative for the epilogue's own
    arithmetic; fp32 layer: 2e-6 relative."""
    R, L, F, E = 300, 128, 256, 64
    dt = torch.float32 if path == "f32" else torch.bfloat16
    cfg = m.LayerConfig(T=R, d_model=L, d_latent=L, n_experts=E, top_k=1, d_ff=F, n_shared=0,
                        d_ff_shared=0, dtype="f32" if path == "f32" else "bf16", pool_rows=320,
                        flags=BF16_PATHS.get(path, 0))
    g = torch.Generator().manual_seed(17)
    w1 = torch.zeros((E, L, F), dtype=dt)
    w3 = torch.zeros((E, L, F), dtype=dt)
    w1[0] = torch.linspace(-30.0, 30.0, L * F)[torch.randperm(L * F, generator=g)].view(L, F)
    w3[0] = torch.linspace(-4.0, 4.0, L * F)[torch.randperm(L * F, generator=g)].view(L, F)
    w2 = (torch.randn((E, F, L), generator=g) * F ** -0.5).to(dt)
    rows = torch.zeros((320, L), dtype=dt)
    rows[torch.arange(R), torch.arange(R) % L] = 1.0
    rows[R:] = float("nan")                                   # padding is never read
    offs = torch.tensor([0] + [R] * E, dtype=torch.int32)     # every row in expert 0
    ws = m.alloc_workspace(cfg, DEV)
    y_perm = torch.zeros((320, L), dtype=dt, device=DEV)
    m.moe_expert_ffn(cfg, rows.to(DEV), offs.to(DEV), w1.to(DEV), w3.to(DEV), w2.to(DEV), y_perm,
                     ws=ws)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(ws)["status"] == 0
    hid = m.workspace_view(ws, cfg, "hidden", dt, (320, F))[:R].double().cpu()
    ref = moe_oracle.swiglu_hidden(rows[:R].double(), w1[0].double(), w3[0].double())
    u1 = w1[0].double()[torch.arange(R) % L]
    assert float(u1.min()) <= -29.9 and float(u1.max()) >= 29.9
    rel = 2e-6 if path == "f32" else 2.0 ** -8 + 2e-5
    err = (hid - ref).abs() - rel * ref.abs()
    worst = int(err.flatten().argmax())
    assert float(err.max()) <= 1e-30, (path, float(hid.flatten()[worst]), float(ref.flatten()[worst]),
                                       float(u1.flatten()[worst]))
    _, o = moe_oracle.grouped_experts(rows[:R], [0, R], w1[:1], w3[:1], w2[:1])
    assert normwise(y_perm[:R], o) <= (1e-5 if path == "f32" else 2e-2)


_PAIR_CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
import sparse_expert_router_gb300 as m
from moe_workloads import SHAPES, make_layer_inputs
from oracle import moe_oracle
for name, T in (("small_bf16", 1000), ("l535b_e64_t1368", 1368)):
    shape = SHAPES[name].with_(T=T)
    cfg = m.LayerConfig.from_shape(shape, flags=m.MOE_FLAG_PDL)
    inp = make_layer_inputs(shape, "cpu")
    dinp = {k: v.to("cuda") for k, v in inp.items()}
    y = torch.empty((T, shape.d_model), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((T, shape.top_k), dtype=torch.int32, device="cuda")
    ws = m.alloc_workspace(cfg)
    m.moe_forward(cfg, dinp, dinp["x"], y, ws, aux={"topk_idx": idx})
    rep = m.moe_get_device_status(ws)
    toks = list(range(0, T, 8))
    ref = moe_oracle.forward(inp, top_k=shape.top_k, rms_eps=shape.rms_eps, tokens=toks)
    assert rep["status"] == 0, rep
    assert torch.equal(idx.cpu().long(), ref["idx"])
    ys = y[toks].double().cpu()
    err = float((ys - ref["y"]).norm() / ref["y"].norm())
    per_row = float(((ys - ref["y"]).norm(dim=1) / ref["y"].norm(dim=1)).max())
    assert err <= 2e-2 and per_row <= 2e-2, (name, err, per_row)
    print(name, "ok", err, per_row)
"""


@pytest.mark.parametrize("env", [{"MOE_TC_PAIR": "0"}, {"MOE_TC_PAIR": "dual"},
                                 {"MOE_TC_PAIR": "glu"}, {"MOE_FRONT_SPLIT": "1"}],
                         ids=["single", "dual", "glu", "front_split"])
def test_pair_modes_forced(env):
    """The tensor-core launches that run as CTA pairs by default (the SwiGLU GEMM 1 and the shared
    experts' gate/up, the grouped dual GEMM 2, the dense dual GEMMs) run on single CTAs instead
    (MOE_TC_PAIR=0), or only the dual ("dual") or SwiGLU ("glu") ones as pairs; or the front GEMMs
    split into the router's launch and a pair launch on layers below the 0.5 TFLOP of front GEMMs
    where that starts by default (MOE_FRONT_SPLIT=1). Each runs in a child process because the
    switches are read once per process; outputs against the oracle, routing exact."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _PAIR_CHILD, root], env=dict(os.environ, **env),
                       cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count(" ok ") == 2, r.stdout


def test_expert_slice():
    """One expert-parallel rank's slice: grouped GEMMs over the active rows of a padded pool,
    then the gate-weighted un-permute back to arrival order."""
    sh = SLICE_C5B
    inp = make_slice_inputs(sh, DEV)
    cfg = m.LayerConfig(T=sh.rows, d_model=sh.d_latent, d_latent=sh.d_latent, n_experts=sh.n_local,
                        top_k=1, d_ff=sh.d_ff, n_shared=0, d_ff_shared=0, dtype=sh.dtype,
                        pool_rows=sh.pool_rows,
                        flags=BF16_PATHS["tc"])
    ws = m.alloc_workspace(cfg, DEV)
    y_perm = torch.full((sh.pool_rows, sh.d_latent), 7.0, dtype=torch.bfloat16, device=DEV)
    m.moe_expert_ffn(cfg, inp["pool"], inp["expert_offsets"], inp["w1"], inp["w3"], inp["w2"],
                     y_perm, ws=ws)
    out = torch.empty((sh.rows, sh.d_latent), dtype=torch.bfloat16, device=DEV)
    m.moe_combine(cfg, y_perm, inp["slot_of"].view(-1, 1), inp["gate"].view(-1, 1), out, ws)
    torch.cuda.synchronize()
    n_act = int(inp["expert_offsets"][-1])
    assert bool((y_perm[n_act:] == 7.0).all())                  # padding never computed
    pos = sample_tokens(sh.rows, 24)
    ref = moe_oracle.slice_rows(inp, pos)
    assert normwise(y_perm[ref["rows"].to(DEV)], ref["y_perm"]) <= 2e-2
    assert normwise(out[pos], ref["out"]) <= 2e-2
    assert m.moe_get_device_status(ws)["status"] == 0


# ------------------------------------------------------- tensor cores vs CUDA cores ----

def test_tc_matches_simt_bitwise_routing_and_close_outputs():
    """The tcgen05 path and the CUDA-core path of the same layer: identical routing (both
    are exact), outputs close (both accumulate in fp32, in different orders)."""
    shape = SHAPES["small_bf16"].with_(T=2048)
    inp = gpu_inputs(shape)
    a = run_forward(shape, inp, BF16_PATHS["tc"])
    b = run_forward(shape, inp, BF16_PATHS["simt"])
    assert torch.equal(a["topk_idx"], b["topk_idx"])
    assert torch.equal(a["slot_of"], b["slot_of"])
    assert normwise(a["y"], b["y"]) <= 1e-2


# ----------------------------------------------------------- programmatic dependent launch ----

def test_pdl_changing_groups_stress():
    """Back-to-back producer -> grouped GEMM launches under programmatic dependent launch with
    the expert group sizes changing on every launch (the hang of the weekly summary of
    2026-09-14, hero-run epic, came from warps that read group boundaries before the producer
    had written them). 50,000 iterations = 100,000 grouped-GEMM launches; the outputs of
    periodic iterations are compared bitwise with the same routing run without PDL."""
    T, d, L, E, k, F = 64, 64, 64, 16, 2, 64
    cfg = m.LayerConfig(T=T, d_model=d, d_latent=L, n_experts=E, top_k=k, d_ff=F, n_shared=0,
                        d_ff_shared=0, dtype="bf16", flags=m.MOE_FLAG_PDL)
    cfg0 = m.LayerConfig(**{**cfg.__dict__, "flags": 0})
    g = torch.Generator().manual_seed(0)
    n_var = 8
    idxs = [torch.stack([torch.randperm(E, generator=g)[:k].sort().values for _ in range(T)])
            .to(torch.int32).to(DEV) for _ in range(n_var)]
    x = torch.randn(T, d, generator=g).to(torch.bfloat16).to(DEV)
    wd = (torch.randn(d, L, generator=g) * d ** -0.5).to(torch.bfloat16).to(DEV)
    gam = torch.ones(L, device=DEV)
    w1 = (torch.randn(E, L, F, generator=g) * L ** -0.5).to(torch.bfloat16).to(DEV)
    w3 = (torch.randn(E, L, F, generator=g) * L ** -0.5).to(torch.bfloat16).to(DEV)
    w2 = (torch.randn(E, F, L, generator=g) * F ** -0.5).to(torch.bfloat16).to(DEV)
    ws = m.alloc_workspace(cfg, DEV)
    bufs = dict(counts=torch.empty(E, dtype=torch.int32, device=DEV),
                offs=torch.empty(E + 1, dtype=torch.int32, device=DEV),
                perm=torch.empty(T * k, dtype=torch.int32, device=DEV),
                slot=torch.empty((T, k), dtype=torch.int32, device=DEV),
                xp=torch.zeros((T * k, L), dtype=torch.bfloat16, device=DEV),
                yp=torch.zeros((T * k, L), dtype=torch.bfloat16, device=DEV))

    def step(c, i):
        b = bufs
        m.moe_permute(c, x, wd, gam, idxs[i % n_var], b["counts"], b["offs"], b["perm"], b["slot"],
                      None, b["xp"], ws)
        m.moe_expert_ffn(c, b["xp"], b["offs"], w1, w3, w2, b["yp"], ws=ws)

    ref = []
    for i in range(n_var):
        step(cfg0, i)
        ref.append(bufs["yp"].clone())
    m.moe_clear_device_status(ws)
    n_iter = 50000
    for i in range(n_iter):
        step(cfg, i)
        if i % 997 == 0 or i == n_iter - 1:
            assert torch.equal(bufs["yp"], ref[i % n_var]), i
    assert m.moe_get_device_status(ws)["status"] == 0


def test_router_logit_error_within_certified_bound():
    """The stage-1 bound the router certifies with, checked on real tensor-core logits: the
    fp32 logits of the router GEMM (at the start of the workspace, after the 256-byte device
    report) against exact fp64 logits. The GEMM accumulates in chunks of 256 k summed in fp32:
    |l~ - l| <= (c g_256 + g_nch (1 + c g_256)) ||x|| ||w_e|| + 2u|l~|, c = 2."""
    from oracle import moe_oracle as O
    for name, c in (("small_bf16", 2.0), ("l535b_t8192", 2.0)):
        shape = SHAPES[name].with_(T=1024)
        inp = gpu_inputs(shape)
        cfg = m.LayerConfig.from_shape(shape)
        ws = m.alloc_workspace(cfg, DEV)
        T, E, d = shape.T, shape.n_experts, shape.d_model
        idx = torch.empty((T, shape.top_k), dtype=torch.int32, device=DEV)
        gate = torch.empty((T, shape.top_k), dtype=torch.float32, device=DEV)
        m.moe_route(cfg, inp["x"], inp["w_router"], inp["b_router"], idx, gate, ws)
        torch.cuda.synchronize()
        lt = ws[256:256 + T * E * 4].view(torch.float32).view(T, E).cpu().double()
        ref, _ = O.router_logits(inp["x"], inp["w_router"], inp["b_router"])
        x64, w64 = O.to64(inp["x"]), O.to64(inp["w_router"])
        u = 2.0 ** -24
        g = lambda n: n * u / (1 - n * u)
        nch = -(-d // 256)
        fac = c * g(256) + g(nch) * (1 + c * g(256))
        beta = fac * x64.norm(dim=1, keepdim=True) * w64.norm(dim=0, keepdim=True) + 2 * u * lt.abs()
        ratio = float(((lt - ref).abs() / beta).max())
        print(name, "max |error| / bound =", ratio)
        assert ratio <= 1.0, ratio


# -------------------------------------------------------------- fp8 expert MLP ----

def _fp8_args(inp, **extra):
    d = {n: inp[n] for n in ("w1_scale", "w3_scale", "w2_scale", "x_scale", "h_scale")}
    d.update(extra)
    return d


def test_small_fp8_forward():
    """fp8 expert MLP (E4M3 rows, hidden and weights): routing bit-exact, outputs against the
    oracle's fp8 layer, the amax outputs bracket the sampled tokens' values."""
    shape = SHAPES["small_fp8"]
    inp = gpu_inputs(shape)
    got = run_forward(shape, inp)
    toks = sample_tokens(shape.T, 256)
    ref = oracle_forward(shape, {k: v.cpu() for k, v in inp.items()}, tokens=toks)
    check_routing(got, ref, shape)
    err = normwise(got["y"][toks], ref["y"])
    assert err <= 2e-2, err
    assert got["report"]["status"] == 0
    # the device's amax runs over every token; the oracle's over the sampled ones
    assert float(got["x_amax"]) >= float(ref["x_amax"]) * (1 - 1e-5)
    assert float(got["h_amax"]) >= float(ref["h_amax"]) * (1 - 1e-4)
    assert float(got["x_amax"]) < 448.0 / float(inp["x_scale"][0])      # no saturation here
    assert float(got["h_amax"]) < 448.0 / float(inp["h_scale"][0])


def test_bf16_expert_ffn_with_shared_experts():
    """moe_expert_ffn on a bf16 layer with the shared experts in the same call: one tensor-core
    launch holds the grouped SwiGLU GEMM and the dense shared one. Both hiddens' SwiGLU
    epilogues hold their results in registers across the accumulator release; y_perm and the
    shared hidden against the oracle, rows past the groups untouched."""
    shape = SHAPES["small_bf16"].with_(T=512)
    cpu = make_layer_inputs(shape, "cpu")
    inp = {k: v.to(DEV) for k, v in cpu.items()}
    cfg = m.LayerConfig.from_shape(shape)
    T, k, L = shape.T, shape.top_k, shape.d_latent
    ref = oracle_forward(shape, cpu)
    R = int(ref["offsets"][-1])
    tok = ref["perm"] // k
    xp = torch.zeros((T * k + 64, L), dtype=torch.bfloat16, device=DEV)
    xp[:R] = ref["h"][tok].to(torch.bfloat16).to(DEV)
    y_perm = torch.zeros((T * k + 64, L), dtype=torch.bfloat16, device=DEV)
    a_s = torch.empty((T, shape.n_shared * shape.d_ff_shared), dtype=torch.bfloat16, device=DEV)
    ws = m.alloc_workspace(cfg, DEV)
    offs = ref["offsets"].to(torch.int32).to(DEV)
    m.moe_expert_ffn(cfg, xp, offs, inp["w1"], inp["w3"], inp["w2"], y_perm, inp["x"],
                     inp["w1_s"], inp["w3_s"], a_s, ws)
    _, o_ref = moe_oracle.grouped_experts(xp[:R].cpu(), ref["offsets"].tolist(), cpu["w1"],
                                          cpu["w3"], cpu["w2"])
    assert normwise(y_perm[:R], o_ref) <= 2e-2
    assert float(y_perm[R:].float().abs().max()) == 0.0
    assert normwise(a_s, ref["a_s"]) <= 2e-2
    assert m.moe_get_device_status(ws)["status"] == 0


def test_fp8_split_calls():
    """moe_permute's E4M3 rows and amax against the oracle's quantization; moe_expert_ffn on the
    oracle's codes (with the shared experts in the same call) and its hidden amax."""
    shape = SHAPES["small_fp8"].with_(T=512)
    cpu = make_layer_inputs(shape, "cpu")
    inp = {k: v.to(DEV) for k, v in cpu.items()}
    cfg = m.LayerConfig.from_shape(shape)
    assert cfg.flags & m.MOE_FLAG_FP8_EXPERTS
    T, k, E, L = shape.T, shape.top_k, shape.n_experts, shape.d_latent
    ref = oracle_forward(shape, cpu)
    sx, sh = float(cpu["x_scale"][0]), float(cpu["h_scale"][0])
    ws = m.alloc_workspace(cfg, DEV)

    oidx = ref["idx"].to(torch.int32).to(DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    slot = torch.empty((T, k), dtype=torch.int32, device=DEV)
    ndrop = torch.empty(1, dtype=torch.int32, device=DEV)
    x_perm = torch.zeros((T * k, L), dtype=torch.uint8, device=DEV)
    x_amax = torch.full((1,), -1.0, device=DEV)
    m.moe_permute(cfg, inp["x"], inp["w_down"], inp["rms_gamma"], oidx, counts, offs, perm, slot,
                  ndrop, x_perm, ws, fp8={"x_scale": inp["x_scale"], "x_amax": x_amax})
    R = int(ref["offsets"][-1])
    assert torch.equal(perm.cpu().long()[:R], ref["perm"])
    tok = ref["perm"] // k
    rows = ref["h"][tok]
    # the device's latent carries fp32 GEMM and norm rounding, well below 1e-3 absolute here
    n_ties = e4m3_codes_match(x_perm[:R].view(torch.float8_e4m3fn).to(torch.float64), rows * sx,
                              atol=1e-3 * sx)
    assert n_ties <= R * L * 1e-3, n_ties
    assert abs(float(x_amax) - float(rows.abs().max())) <= 1e-5 * float(rows.abs().max())

    # the oracle's codes as the grouped rows; 64 rows past the pool are never touched
    codes = moe_oracle.quantize_e4m3(rows, sx)
    xp = torch.zeros((T * k + 64, L), dtype=torch.uint8, device=DEV)
    xp[:R] = codes.to(torch.float8_e4m3fn).view(torch.uint8).to(DEV)
    y_perm = torch.zeros((T * k + 64, L), dtype=torch.bfloat16, device=DEV)
    a_s = torch.empty((T, shape.n_shared * shape.d_ff_shared), dtype=torch.bfloat16, device=DEV)
    h_amax = torch.full((1,), -1.0, device=DEV)
    m.moe_expert_ffn(cfg, xp, ref["offsets"].to(torch.int32).to(DEV), inp["w1"], inp["w3"],
                     inp["w2"], y_perm, inp["x"], inp["w1_s"], inp["w3_s"], a_s, ws,
                     fp8=_fp8_args(inp, h_amax=h_amax))
    a_ref, o_ref = moe_oracle.grouped_experts(
        codes, ref["offsets"].tolist(), cpu["w1"], cpu["w3"], cpu["w2"],
        fp8={n: cpu[n] for n in ("w1_scale", "w3_scale", "w2_scale", "x_scale", "h_scale")})
    assert normwise(y_perm[:R], o_ref) <= 1e-2
    assert float(y_perm[R:].float().abs().max()) == 0.0
    assert normwise(a_s, ref["a_s"]) <= 1e-2
    hmax = float(a_ref.abs().max())
    assert abs(float(h_amax) - hmax) <= 1e-4 * hmax, (float(h_amax), hmax)
    # an fp8 layer without its moe_fp8_t is an argument error, not a fault
    with pytest.raises(m.MoEError):
        m.moe_expert_ffn(cfg, xp, offs, inp["w1"], inp["w3"], inp["w2"], y_perm, ws=ws)
    with pytest.raises(m.MoEError):
        m.moe_permute(cfg, inp["x"], inp["w_down"], inp["rms_gamma"], oidx, counts, offs, perm,
                      slot, ndrop, x_perm, ws)
    assert m.moe_get_device_status(ws)["status"] == 0


def test_fp8_close_to_bf16_layer():
    """The fp8 layer and the bf16 layer with the same weights (dequantized, exact in bf16):
    identical routing, outputs apart by no more than E4M3 activation rounding allows (each
    quantized value is within 2^-4 of its input, relatively), and not identical."""
    shape = SHAPES["small_fp8"].with_(T=2048)
    inp = gpu_inputs(shape)
    a = run_forward(shape, inp)
    deq = dict(inp)
    for n in ("w1", "w3", "w2"):
        deq[n] = (inp[n].float() * inp[n + "_scale"].unsqueeze(1)).to(torch.bfloat16)
    b = run_forward(shape.with_(expert_dtype="bf16"), deq)
    assert torch.equal(a["topk_idx"], b["topk_idx"])
    assert torch.equal(a["expert_offsets"], b["expert_offsets"])
    err = normwise(a["y"], b["y"])
    assert 1e-3 < err <= 0.1, err


# --------------------------------------------------------- attention-mask padding ----

@pytest.mark.parametrize("cap", [None, (1, 2)], ids=["nocap", "cf050"])
def test_token_mask_tiny_f32(cap):
    """Padding tokens excluded from dispatch: every output against the oracle, and moe_permute
    with the same mask writes the same slots."""
    shape = SHAPES["tiny_f32"].with_(capacity=cap)
    cpu = make_layer_inputs(shape, "cpu")
    inp = {k: v.to(DEV) for k, v in cpu.items()}
    mask = padding_mask(shape.T, seq_len=32, seed=1)
    assert 0 < int(mask.sum()) < shape.T
    got = run_forward(shape, inp, token_mask=mask)
    ref = oracle_forward(shape, dict(cpu, token_mask=mask))
    check_routing(got, ref, shape)
    assert bool((got["slot_of"].cpu()[mask == 0] == -1).all())
    err = normwise(got["y"], ref["y"])
    assert err <= 1e-5, err
    assert got["report"]["status"] == 0
    # the split call with the mask
    T, k, E, L = shape.T, shape.top_k, shape.n_experts, shape.d_latent
    cfg = m.LayerConfig.from_shape(shape)
    ws = m.alloc_workspace(cfg, DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    slot = torch.empty((T, k), dtype=torch.int32, device=DEV)
    ndrop = torch.empty(1, dtype=torch.int32, device=DEV)
    x_perm = torch.zeros((T * k, L), dtype=torch.float32, device=DEV)
    m.moe_permute(cfg, inp["x"], inp["w_down"], inp["rms_gamma"],
                  ref["idx"].to(torch.int32).to(DEV), counts, offs, perm, slot, ndrop, x_perm, ws,
                  token_mask=mask.to(DEV))
    assert torch.equal(slot.cpu().long(), ref["slot_of"])
    assert torch.equal(counts.cpu().long(), ref["counts"])
    assert int(ndrop.cpu()) == int(ref["n_dropped"])


def test_token_mask_small_bf16():
    shape = SHAPES["small_bf16"].with_(T=2048, capacity=(11, 10))
    inp = gpu_inputs(shape)
    mask = padding_mask(shape.T, seq_len=256, seed=2)
    got = run_forward(shape, inp, token_mask=mask)
    pads = (mask == 0).nonzero().flatten()[:6].tolist()
    toks = sample_tokens(shape.T, 96, extra=pads)
    ref = oracle_forward(shape, dict({k: v.cpu() for k, v in inp.items()}, token_mask=mask),
                         tokens=toks)
    check_routing(got, ref, shape)
    err = normwise(got["y"][toks], ref["y"])
    assert err <= 2e-2, err
    assert got["report"]["status"] == 0


def test_fp8_with_capacity_and_padding():
    """fp8 experts together with a capacity that drops assignments and attention-mask padding:
    routing, drops and slots bit-exact, outputs (dropped and padding tokens included) against
    the oracle's fp8 layer."""
    shape = SHAPES["small_fp8"].with_(T=2048, capacity=(1, 2))
    inp = gpu_inputs(shape)
    mask = padding_mask(shape.T, seq_len=256, seed=4)
    got = run_forward(shape, inp, token_mask=mask)
    pads = (mask == 0).nonzero().flatten()[:6].tolist()
    dropped = (got["slot_of"].cpu() < 0).any(1).nonzero().flatten()
    dropped = [t for t in dropped.tolist() if int(mask[t])][:6]
    toks = sample_tokens(shape.T, 64, extra=pads + dropped)
    ref = oracle_forward(shape, dict({k: v.cpu() for k, v in inp.items()}, token_mask=mask),
                         tokens=toks)
    check_routing(got, ref, shape)
    assert int(ref["n_dropped"]) > 0 and len(dropped) > 0
    err = normwise(got["y"][toks], ref["y"])
    assert err <= 2e-2, err
    assert got["report"]["status"] == 0


# ---------------------------------------------------------- expert MLP backward ----

def _backward_case(E, L, F, counts, seed=21, pad=64):
    """bf16 grouped rows (expert-major, ragged groups with empty experts and tails that are not
    multiples of 64 rows), weights and an output gradient; the pool's padding rows hold NaN so
    that anything read past the groups shows."""
    g = torch.Generator().manual_seed(seed)
    R = sum(counts)
    offs = [0]
    for c in counts:
        offs.append(offs[-1] + c)
    P = R + pad
    x = torch.full((P, L), float("nan"))
    x[:R] = torch.randn(R, L, generator=g)
    dy = torch.full((P, L), float("nan"))
    dy[:R] = torch.randn(R, L, generator=g)
    w1 = torch.randn(E, L, F, generator=g) * L ** -0.5
    w3 = torch.randn(E, L, F, generator=g) * L ** -0.5
    w2 = torch.randn(E, F, L, generator=g) * F ** -0.5
    bf = lambda t: t.to(torch.bfloat16)
    return {"x": bf(x), "dy": bf(dy), "w1": bf(w1), "w3": bf(w3), "w2": bf(w2), "offs": offs,
            "P": P, "R": R}


def _run_backward(c, E, L, F):
    cfg = m.LayerConfig(T=c["P"], d_model=L, d_latent=L, n_experts=E, top_k=1, d_ff=F,
                        n_shared=0, d_ff_shared=0, dtype="bf16", pool_rows=c["P"])
    ws = m.alloc_backward_workspace(cfg, DEV)
    d = {n: c[n].to(DEV) for n in ("x", "dy", "w1", "w3", "w2")}
    offs = torch.tensor(c["offs"], dtype=torch.int32, device=DEV)
    out = {"dx": torch.full((c["P"], L), 3.0, dtype=torch.bfloat16, device=DEV),
           "dw1": torch.full((E, L, F), 5.0, dtype=torch.bfloat16, device=DEV),
           "dw3": torch.full((E, L, F), 5.0, dtype=torch.bfloat16, device=DEV),
           "dw2": torch.full((E, F, L), 5.0, dtype=torch.bfloat16, device=DEV)}
    m.moe_expert_ffn_backward(cfg, d["x"], offs, d["w1"], d["w3"], d["w2"], d["dy"], out["dx"],
                              out["dw1"], out["dw3"], out["dw2"], ws)
    torch.cuda.synchronize()
    out["report"] = m.moe_get_device_status(ws)
    return out


@pytest.mark.parametrize("E,L,F,counts", [
    (6, 256, 384, (70, 0, 129, 1, 64, 200)),
    (8, 1024, 1024, (171, 333, 0, 17, 256, 97, 0, 512)),
], ids=["ragged_small", "ragged_1024"])
def test_expert_backward(E, L, F, counts):
    """dx_perm and every weight gradient against the oracle's chain rule; rows past the groups
    untouched; experts without rows get exact zeros."""
    c = _backward_case(E, L, F, counts)
    got = _run_backward(c, E, L, F)
    ref = moe_oracle.grouped_experts_backward(c["x"][:c["R"]], c["offs"], c["w1"], c["w3"],
                                              c["w2"], c["dy"][:c["R"]])
    R = c["R"]
    assert got["report"]["status"] == 0
    assert normwise(got["dx"][:R], ref["dx"]) <= 2e-2
    assert bool((got["dx"][R:].float() == 3.0).all())
    for n in ("dw1", "dw3", "dw2"):
        g = got[n].float()
        assert not bool(torch.isnan(g).any()), n
        err = normwise(g, ref[n])
        assert err <= 2e-2, (n, err)
        for e, cnt in enumerate(counts):
            if cnt == 0:
                assert float(g[e].abs().max()) == 0.0, (n, e)


def _many_expert_counts(E=320):
    """Rows per expert for a grouped problem large enough that the weight-gradient kernel gives
    each work unit several m tiles: empty experts, groups of 1-4 k steps with tails (their b
    tile stays in shared memory across the unit's m tiles) and groups above 256 rows (b
    streamed)."""
    counts = []
    for e in range(E):
        if e % 10 == 0:
            counts.append(0)
        elif e % 16 == 3:
            counts.append(257 + (e * 37) % 200)
        elif e % 5 == 1:
            counts.append(193 + (e * 13) % 64)
        elif e % 9 == 4:
            counts.append(129 + (e * 11) % 64)
        else:
            counts.append(1 + (e * 29) % 128)
    return tuple(counts)


def test_expert_backward_many_experts():
    """320 experts, L = F = 512: the weight-gradient units hold 2 m tiles each, so a resident b
    tile serves two accumulators; gradients against the oracle, empty experts exactly zero."""
    E, L, F = 320, 512, 512
    counts = _many_expert_counts(E)
    c = _backward_case(E, L, F, counts, seed=9)
    got = _run_backward(c, E, L, F)
    ref = moe_oracle.grouped_experts_backward(c["x"][:c["R"]], c["offs"], c["w1"], c["w3"],
                                              c["w2"], c["dy"][:c["R"]])
    assert got["report"]["status"] == 0
    assert normwise(got["dx"][:c["R"]], ref["dx"]) <= 2e-2
    for n in ("dw1", "dw3", "dw2"):
        g = got[n].float()
        err = normwise(g, ref[n])
        assert err <= 2e-2, (n, err)
        # per-expert check as well: a wrong m tile or unit shows in a single expert
        for e in range(0, E, 7):
            if counts[e]:
                assert normwise(g[e], ref[n][e]) <= 3e-2, (n, e, counts[e])
        zero = [e for e, cnt in enumerate(counts) if cnt == 0]
        assert float(g[zero].abs().max()) == 0.0, n


def test_expert_backward_deterministic():
    """Two runs give bitwise equal gradients (fixed accumulation order, no atomics)."""
    E, L, F, counts = 4, 256, 256, (100, 37, 0, 300)
    c = _backward_case(E, L, F, counts, seed=5)
    a = _run_backward(c, E, L, F)
    b = _run_backward(c, E, L, F)
    for n in ("dx", "dw1", "dw3", "dw2"):
        assert torch.equal(a[n].view(torch.int16), b[n].view(torch.int16)), n


# ---------------------------------------------------------------- layer backward ----

def _layer_grads(shape, inp):
    E, L, F, d = shape.n_experts, shape.d_latent, shape.d_ff, shape.d_model
    S, Fs = shape.n_shared, shape.d_ff_shared
    bf = dict(dtype=torch.bfloat16, device=DEV)
    return {"dw_router": torch.full((d, E), 9.0, **bf),
            "db_router": torch.full((E,), 9.0, dtype=torch.float32, device=DEV),
            "dw_down": torch.full((d, L), 9.0, **bf),
            "drms_gamma": torch.full((L,), 9.0, dtype=torch.float32, device=DEV),
            "dw1": torch.full((E, L, F), 9.0, **bf), "dw3": torch.full((E, L, F), 9.0, **bf),
            "dw2": torch.full((E, F, L), 9.0, **bf), "dw1_s": torch.full((S, d, Fs), 9.0, **bf),
            "dw3_s": torch.full((S, d, Fs), 9.0, **bf), "dw2_s": torch.full((S, Fs, d), 9.0, **bf),
            "dw_up": torch.full((L, d), 9.0, **bf)}


@pytest.mark.parametrize("cap,masked", [(None, False), ((1, 1), False), (None, True)],
                         ids=["nocap", "cf100", "padding"])
def test_layer_backward(cap, masked):
    """dx and every weight gradient of the whole layer against the oracle's chain rule, after
    the forward on the same inputs (with capacity drops, or with padding tokens)."""
    shape = SHAPES["small_bf16"].with_(T=512, capacity=cap)
    cpu = make_layer_inputs(shape, "cpu")
    if masked:
        cpu["token_mask"] = padding_mask(shape.T, seq_len=128, seed=5)
    inp = {k: v.to(DEV) for k, v in cpu.items()}
    cfg = m.LayerConfig.from_shape(shape)
    T, d = shape.T, shape.d_model
    fws = m.alloc_workspace(cfg, DEV)
    y = torch.empty((T, d), dtype=torch.bfloat16, device=DEV)
    m.moe_forward(cfg, inp, inp["x"], y, fws,
                  aux={"token_mask": inp["token_mask"]} if masked else None)
    g = torch.Generator().manual_seed(3)
    dy = torch.randn(T, d, generator=g).to(torch.bfloat16)
    dx = torch.full((T, d), 9.0, dtype=torch.bfloat16, device=DEV)
    grads = _layer_grads(shape, inp)
    bws = m.alloc_layer_backward_workspace(cfg, DEV)
    m.moe_backward(cfg, inp, inp["x"], dy.to(DEV), dx, grads, fws, bws)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(bws)["status"] == 0
    fwd = oracle_forward(shape, cpu)
    if cap:
        assert int(fwd["n_dropped"]) > 0
    ref = moe_oracle.backward(cpu, fwd, dy, rms_eps=shape.rms_eps)
    errs = {"dx": normwise(dx, ref["dx"])}
    for n in grads:
        errs[n] = normwise(grads[n].float(), ref[n])
    bad = {n: e for n, e in errs.items() if not e <= 2e-2}
    assert not bad, (bad, errs)


def test_expert_backward_full_size_sampled():
    """The routed experts' backward at the 535B layer's full size, in the launch configuration the
    bench times (the workload's own routing, PDL on; 24 m tiles per weight-gradient work unit):
    the weight gradients of three experts (the largest group, a middle one and the smallest
    non-empty one) and their rows' dx against the oracle's chain rule for those experts alone."""
    shape = SHAPES["l535b_t8192"]
    cfg = m.LayerConfig.from_shape(shape, flags=m.MOE_FLAG_PDL)
    T, k, E, L = shape.T, shape.top_k, shape.n_experts, shape.d_latent
    inp = make_layer_inputs(shape, DEV)
    ws = m.alloc_workspace(cfg, DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, k), dtype=torch.float32, device=DEV)
    m.moe_route(cfg, inp["x"], inp["w_router"], inp["b_router"], idx, gate, ws)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    slot = torch.empty((T, k), dtype=torch.int32, device=DEV)
    ndrop = torch.empty(1, dtype=torch.int32, device=DEV)
    xp = torch.empty((T * k, L), dtype=torch.bfloat16, device=DEV)
    m.moe_permute(cfg, inp["x"], inp["w_down"], inp["rms_gamma"], idx, counts, offs, perm, slot,
                  ndrop, xp, ws)
    g = torch.Generator(device=DEV).manual_seed(7)
    dy = torch.randn((T * k, L), generator=g, device=DEV).to(torch.bfloat16)
    dx = torch.empty_like(xp)
    dw1, dw3, dw2 = (torch.empty_like(inp[n]) for n in ("w1", "w3", "w2"))
    bws = m.alloc_backward_workspace(cfg, DEV)
    m.moe_expert_ffn_backward(cfg, xp, offs, inp["w1"], inp["w3"], inp["w2"], dy, dx, dw1, dw3,
                              dw2, bws)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(bws)["status"] == 0
    c, o = counts.cpu(), offs.cpu()
    nz = (c > 0).nonzero().flatten()
    order = nz[c[nz].argsort()]
    for e in (int(order[-1]), int(order[len(order) // 2]), int(order[0])):
        lo, hi = int(o[e]), int(o[e + 1])
        ref = moe_oracle.grouped_experts_backward(xp[lo:hi], [0, hi - lo], inp["w1"][e:e + 1],
                                                  inp["w3"][e:e + 1], inp["w2"][e:e + 1],
                                                  dy[lo:hi])
        for n, got in (("dw1", dw1[e]), ("dw3", dw3[e]), ("dw2", dw2[e])):
            err = normwise(got.float(), ref[n][0])
            assert err <= 2e-2, (n, e, hi - lo, err)
        assert normwise(dx[lo:hi], ref["dx"]) <= 2e-2, (e, hi - lo)
    del inp, dw1, dw3, dw2
    torch.cuda.empty_cache()


def test_layer_backward_full_size_sampled_dx():
    """The whole layer's backward at the 535B layer's full size (PDL on, as the bench times it):
    dx of sampled tokens against the oracle's chain rule on those tokens alone. A token's dx
    depends only on its own row, and without a capacity its routing is its own."""
    shape = SHAPES["l535b_t8192"]
    cfg = m.LayerConfig.from_shape(shape, flags=m.MOE_FLAG_PDL)
    T, d, L, E = shape.T, shape.d_model, shape.d_latent, shape.n_experts
    inp = make_layer_inputs(shape, DEV)
    fws = m.alloc_workspace(cfg, DEV)
    y = torch.empty((T, d), dtype=torch.bfloat16, device=DEV)
    m.moe_forward(cfg, inp, inp["x"], y, fws)
    g = torch.Generator(device=DEV).manual_seed(7)
    dy = torch.randn((T, d), generator=g, device=DEV).to(torch.bfloat16)
    dx = torch.empty((T, d), dtype=torch.bfloat16, device=DEV)
    grads = {n: torch.empty_like(inp[n[1:]]) for n in m.GRAD_NAMES
             if n not in ("db_router", "drms_gamma")}
    grads["db_router"] = torch.empty(E, dtype=torch.float32, device=DEV)
    grads["drms_gamma"] = torch.empty(L, dtype=torch.float32, device=DEV)
    bws = m.alloc_layer_backward_workspace(cfg, DEV)
    m.moe_backward(cfg, inp, inp["x"], dy, dx, grads, fws, bws)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(bws)["status"] == 0
    toks = sample_tokens(T, 4)
    sub = dict(inp)
    sub["x"] = inp["x"][toks]
    fwd = moe_oracle.forward(sub, top_k=shape.top_k, rms_eps=shape.rms_eps)
    ref = moe_oracle.backward(sub, fwd, dy[toks], rms_eps=shape.rms_eps, expert_weight_grads=False)
    err = normwise(dx[toks], ref["dx"])
    assert err <= 2e-2, err
    del inp, grads
    torch.cuda.empty_cache()


# -------------------------------------------------------------------- edge cases ----

from moe_workloads import LayerShape  # noqa: E402

EDGE = {
    # one token; every stage runs on a single row
    "t1_f32": (LayerShape("t1_f32", T=1, d_model=256, d_latent=128, n_experts=16, top_k=2,
                          d_ff=128, n_shared=1, d_ff_shared=256, dtype="f32"), 0),
    "t1_bf16": (LayerShape("t1_bf16", T=1, d_model=256, d_latent=128, n_experts=64, top_k=8,
                           d_ff=128, n_shared=1, d_ff_shared=256, dtype="bf16"), 0),
    # k = E: every expert selected, gates = the full softmax
    "k_eq_e": (LayerShape("k_eq_e", T=257, d_model=256, d_latent=128, n_experts=16, top_k=16,
                          d_ff=128, n_shared=1, d_ff_shared=256, dtype="f32"), 0),
    # k = 1 with a capacity of one row per expert and ragged token count
    "k1_cap": (LayerShape("k1_cap", T=333, d_model=256, d_latent=128, n_experts=16, top_k=1,
                          d_ff=128, n_shared=1, d_ff_shared=256, dtype="f32",
                          capacity=(1, 21)), 0),
    # the limits: 1024 experts, top-32, ragged T on the tensor-core path
    "e1024_k32": (LayerShape("e1024_k32", T=300, d_model=256, d_latent=128, n_experts=1024,
                             top_k=32, d_ff=128, n_shared=0, d_ff_shared=0, dtype="bf16"), 0),
    "e1024_k32_simt": (LayerShape("e1024_k32_simt", T=129, d_model=256, d_latent=128,
                                  n_experts=1024, top_k=32, d_ff=128, n_shared=0, d_ff_shared=0,
                                  dtype="bf16"), m.MOE_FLAG_SIMT),
    # no shared experts, latent == model width, T one past a 256-row token tile
    "no_shared": (LayerShape("no_shared", T=257, d_model=128, d_latent=128, n_experts=64,
                             top_k=4, d_ff=256, n_shared=0, d_ff_shared=0, dtype="bf16"), 0),
    # the fp8 expert path at the same edges: one token (most experts empty, one-row groups),
    # 1024 experts with top-32 (groups of ~9 rows), k = 1 with capacity 1 per expert
    "t1_fp8": (LayerShape("t1_fp8", T=1, d_model=256, d_latent=128, n_experts=64, top_k=8,
                          d_ff=128, n_shared=1, d_ff_shared=256, dtype="bf16",
                          expert_dtype="fp8"), 0),
    "e1024_k32_fp8": (LayerShape("e1024_k32_fp8", T=300, d_model=256, d_latent=128,
                                 n_experts=1024, top_k=32, d_ff=128, n_shared=0, d_ff_shared=0,
                                 dtype="bf16", expert_dtype="fp8"), 0),
    "k1_cap_fp8": (LayerShape("k1_cap_fp8", T=333, d_model=256, d_latent=128, n_experts=64,
                              top_k=1, d_ff=128, n_shared=1, d_ff_shared=256, dtype="bf16",
                              capacity=(1, 21), expert_dtype="fp8"), 0),
    # widths at which the expert GEMMs run as CTA pairs (d_ff a multiple of 256, d_latent of
    # 512), bf16 and fp8, with one-row and empty groups (T = 1) and ~9-row groups (E = 1024)
    "t1_pair": (LayerShape("t1_pair", T=1, d_model=512, d_latent=512, n_experts=64, top_k=8,
                           d_ff=256, n_shared=1, d_ff_shared=256, dtype="bf16"), 0),
    "t1_pair_fp8": (LayerShape("t1_pair_fp8", T=1, d_model=512, d_latent=512, n_experts=64,
                               top_k=8, d_ff=256, n_shared=1, d_ff_shared=256, dtype="bf16",
                               expert_dtype="fp8"), 0),
    "e1024_pair_fp8": (LayerShape("e1024_pair_fp8", T=300, d_model=512, d_latent=512,
                                  n_experts=1024, top_k=32, d_ff=256, n_shared=0, d_ff_shared=0,
                                  dtype="bf16", expert_dtype="fp8"), 0),
}


@pytest.mark.parametrize("pdl", list(PDL_FLAGS))
@pytest.mark.parametrize("name", list(EDGE))
def test_edge_case_forward(name, pdl):
    """Every token's routing, dispatch and output against the oracle at the edges the method
    allows: a single token, k = E, k = 1 with capacity 1, 1024 experts with top-32, no shared
    experts, token counts one past a tile; the fp8 expert path at three of them; and the CTA-pair
    expert GEMMs (bf16 and fp8) with one-row, empty and ~9-row groups."""
    shape, flags = EDGE[name]
    cpu = make_layer_inputs(shape, "cpu")
    inp = {k: v.to(DEV) for k, v in cpu.items()}
    got = run_forward(shape, inp, flags | PDL_FLAGS[pdl])
    ref = oracle_forward(shape, cpu)
    check_routing(got, ref, shape)
    if shape.capacity:
        assert int(ref["n_dropped"]) > 0
    if shape.top_k == shape.n_experts:
        assert torch.equal(got["topk_idx"].cpu(), torch.arange(shape.n_experts, dtype=torch.int32)
                           .expand(shape.T, -1))
    err = normwise(got["y"], ref["y"])
    assert err <= (1e-5 if shape.dtype == "f32" else 2e-2), err
    assert got["report"]["status"] == 0


@pytest.mark.parametrize("name", ["tiny_f32", "small_bf16", "small_fp8"])
def test_forward_cuda_graph_replay(name):
    """moe_forward captured in a CUDA graph (PDL edges included) and replayed on new inputs
    copied into the captured buffer gives the bits of an eager call on the same inputs."""
    shape = SHAPES[name]
    inp = gpu_inputs(shape)
    flags = m.MOE_FLAG_PDL
    cfg = m.LayerConfig.from_shape(shape, flags=flags)
    T, d = shape.T, shape.d_model
    ws = m.alloc_workspace(cfg, DEV)
    x = inp["x"].clone()
    y = torch.empty((T, d), dtype=shape.torch_dtype, device=DEV)
    st = torch.cuda.Stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(m.MOE_FORWARD_STAGES + 1)]
    for e in evs:
        e.record(st)
    aux = {"stage_events": evs}
    with torch.cuda.stream(st):
        m.moe_forward(cfg, inp, x, y, ws, stream=st, aux=aux)   # first call outside the capture
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        m.moe_forward(cfg, inp, x, y, ws, stream=st, aux=aux)
    gen = torch.Generator().manual_seed(9)
    for _ in range(3):
        xn = torch.randn(T, d, generator=gen).to(shape.torch_dtype).to(DEV)
        x.copy_(xn)
        g.replay()
        evs[-1].synchronize()                                   # the stage events are replayed too
        assert evs[0].elapsed_time(evs[-1]) > 0
        torch.cuda.synchronize()
        y_graph = y.clone()
        y_eager = torch.empty_like(y)
        m.moe_forward(cfg, inp, xn, y_eager, ws)
        torch.cuda.synchronize()
        bits = torch.int16 if shape.dtype == "bf16" else torch.int32
        assert torch.equal(y_graph.view(bits), y_eager.view(bits))
    assert m.moe_get_device_status(ws)["status"] == 0


@pytest.mark.parametrize("name", ["small_bf16", "small_fp8"])
def test_forward_pipelined_matches_forward(name):
    """The host-buffer serving path gives, batch for batch, the bits moe_forward gives."""
    shape = SHAPES[name].with_(T=512)
    inp = gpu_inputs(shape)
    cfg = m.LayerConfig.from_shape(shape, flags=m.MOE_FLAG_PDL)
    T, d = shape.T, shape.d_model
    g = torch.Generator().manual_seed(4)
    xs = [torch.randn(T, d, generator=g).to(torch.bfloat16).pin_memory() for _ in range(5)]
    ys = [torch.empty(T, d, dtype=torch.bfloat16).pin_memory() for _ in range(5)]
    ws = m.alloc_workspace(cfg, DEV)
    x_stage = torch.empty((2, T, d), dtype=torch.bfloat16, device=DEV)
    y_stage = torch.empty((2, T, d), dtype=torch.bfloat16, device=DEV)
    st, h2d, d2h = torch.cuda.current_stream(), torch.cuda.Stream(), torch.cuda.Stream()
    m.moe_forward_pipelined(cfg, inp, xs, ys, x_stage, y_stage, ws, st, h2d, d2h)
    st.synchronize()
    for i in range(5):
        y = torch.empty((T, d), dtype=torch.bfloat16, device=DEV)
        m.moe_forward(cfg, inp, xs[i].to(DEV), y, ws)
        torch.cuda.synchronize()
        assert torch.equal(ys[i].view(torch.int16), y.cpu().view(torch.int16)), i
    with pytest.raises(m.MoEError):      # the three streams must differ
        m.moe_forward_pipelined(cfg, inp, xs, ys, x_stage, y_stage, ws, st, h2d, h2d)
