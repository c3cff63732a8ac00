"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Some callers of this library may not allocate: an allocator-free runtime or plugin that only
receives its input and output buffers, or code that must not call cudaMalloc while other work
is in flight. moe_route_noalloc serves them with a fixed scratch array inside the library
instead of a caller workspace. These tests call it through the C ABI and check its results
against moe_route (the entry point that takes a workspace) on two calls in a row, so that the
second call runs on scratch the first one left behind. This file is collected last on purpose.
"""
import pytest
import torch

import sparse_expert_router_gb300 as m
from gpu_cases import near_tie_router
from moe_workloads import SHAPES, make_router_inputs
from oracle import moe_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _route_both(shape, flags):
    cfg = m.LayerConfig.from_shape(shape, flags=flags)
    inp = make_router_inputs(shape, DEV)
    T, k = shape.T, shape.top_k
    idx_ref = torch.empty((T, k), dtype=torch.int32, device=DEV)
    gate_ref = torch.empty((T, k), dtype=torch.float32, device=DEV)
    ws = m.alloc_workspace(cfg, DEV)
    m.moe_route(cfg, inp["x"], inp["w_router"], inp["b_router"], idx_ref, gate_ref, ws)
    idx = torch.full((T, k), -1, dtype=torch.int32, device=DEV)
    gate = torch.zeros((T, k), dtype=torch.float32, device=DEV)
    report = torch.full((4,), -1, dtype=torch.int32, device=DEV)
    m.moe_route_noalloc(cfg, inp["x"], inp["w_router"], inp["b_router"], idx, gate, report)
    torch.cuda.synchronize()
    return idx_ref, gate_ref, idx, gate, report.cpu().tolist(), m.moe_get_device_status(ws)


@pytest.mark.parametrize("name,flags", [("l535b_t8192", 0), ("small_bf16", m.MOE_FLAG_SIMT),
                                        ("tiny_f32", 0)])
def test_noalloc_matches_moe_route_on_two_calls(name, flags):
    tol = 1e-6 if SHAPES[name].dtype == "f32" else 1e-5
    for call, seed in enumerate((11, 12)):            # two calls in a row, different tokens
        shape = SHAPES[name].with_(seed=seed, T=SHAPES[name].T // (call + 1))
        idx_ref, gate_ref, idx, gate, rep, rep_ref = _route_both(shape, flags)
        assert torch.equal(idx, idx_ref), (name, call)
        assert float((gate - gate_ref).abs().max()) <= tol, (name, call)
        assert rep[0] == 0, rep
        assert rep[2] == rep_ref["n_refined"] and rep[3] == rep_ref["n_exact"], (rep, rep_ref)


def test_noalloc_exact_stage_on_near_ties():
    """Inputs where nearly every token needs exact logits (more than the 64 tokens whose stage-2
    state the library hands to the exact stage), on scratch left behind by a previous call:
    indices equal to the oracle's exact top-k and to moe_route's."""
    x, w = near_tie_router(T=512)
    T, d = x.shape
    E, k = w.shape[1], 8
    cfg = m.LayerConfig(T=T, d_model=d, d_latent=64, n_experts=E, top_k=k, d_ff=64, n_shared=0,
                        d_ff_shared=0, dtype="bf16")
    idx = torch.full((T, k), -1, dtype=torch.int32, device=DEV)
    gate = torch.zeros((T, k), dtype=torch.float32, device=DEV)
    report = torch.full((4,), -1, dtype=torch.int32, device=DEV)
    m.moe_route_noalloc(cfg, x.to(DEV), w.to(DEV), None, idx, gate, report)
    torch.cuda.synchronize()
    rep = report.cpu().tolist()
    ref = moe_oracle.route(x, w, None, k)
    assert torch.equal(idx.cpu().long(), ref["idx"])
    assert rep[0] == 0 and rep[3] > 64, rep
    ws = m.alloc_workspace(cfg, DEV)
    idx2 = torch.empty_like(idx)
    m.moe_route(cfg, x.to(DEV), w.to(DEV), None, idx2, torch.empty_like(gate), ws)
    assert torch.equal(idx, idx2)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    shape = SHAPES["l535b_t65536"]                    # 65,536 x 384 fp32 logits alone exceed 32 MiB
    cfg = m.LayerConfig.from_shape(shape)
    x = torch.zeros((8, 8), dtype=torch.bfloat16, device=DEV)   # never read: rejected up front
    out = torch.zeros((8, 8), dtype=torch.int32, device=DEV)
    with pytest.raises(m.MoEError) as e:
        m.moe_route_noalloc(cfg, x, x, None, out, out.float())
    assert e.value.status == 3                        # MOE_ERR_WORKSPACE
