"""The C-ABI library: loads without a GPU, exports every declared symbol, and rejects bad
arguments with status codes before touching the device (CPU only)."""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def lib():
    from sparse_expert_router_gb300.build import build_library
    build_library()
    import sparse_expert_router_gb300 as m
    return m.load()


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)))


def test_header_declares_api():
    names = declared_functions()
    for n in ("moe_route", "moe_permute", "moe_expert_ffn", "moe_combine", "moe_forward",
              "moe_workspace_size", "moe_get_device_status"):
        assert n in names


def test_exports_every_declared_symbol(lib):
    from sparse_expert_router_gb300 import _lib
    path = _lib.LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (moe_\w+)", out))
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(lib, n)
    # nothing else of ours leaks out of the library
    assert exported == set(declared_functions())
    # the binding wraps every declared entry point under the same name
    assert set(_lib.SIGNATURES) == set(declared_functions())


def _cfg(**kw):
    import sparse_expert_router_gb300 as m
    base = dict(T=256, d_model=256, d_latent=128, n_experts=16, top_k=2, d_ff=128, n_shared=1,
                d_ff_shared=256, dtype="f32")
    base.update(kw)
    return m.LayerConfig(**base)


def _ws(lib, cfg):
    n = C.c_size_t(0)
    assert lib.moe_workspace_size(C.byref(cfg.c()), C.byref(n)) == 0
    return n.value


def test_workspace_size_and_config_errors(lib):
    from sparse_expert_router_gb300 import _lib as L
    n = _ws(lib, _cfg())
    assert n > 0 and n % 256 == 0
    assert _ws(lib, _cfg(T=512)) > n
    bad = [(dict(top_k=17), L.MOE_ERR_INVALID_ARG), (dict(T=0), L.MOE_ERR_INVALID_ARG),
           (dict(n_experts=2048, top_k=2), L.MOE_ERR_UNSUPPORTED),
           (dict(top_k=33, n_experts=64), L.MOE_ERR_UNSUPPORTED),
           (dict(d_model=250), L.MOE_ERR_ALIGNMENT),
           (dict(capacity=(11, 0)), L.MOE_ERR_INVALID_ARG)]
    for kw, code in bad:
        c = _cfg(**kw)
        assert lib.moe_workspace_size(C.byref(c.c()), C.byref(C.c_size_t())) == code, kw
    assert lib.moe_workspace_size(None, C.byref(C.c_size_t())) == L.MOE_ERR_INVALID_ARG


def test_argument_errors_before_any_launch(lib):
    """Fake but aligned pointers: every call must fail validation without dereferencing them."""
    from sparse_expert_router_gb300 import _lib as L
    cfg = _cfg()
    c = C.byref(cfg.c())
    n = _ws(lib, cfg)
    P = lambda v: C.c_void_p(v)
    good, odd, ws = P(0x10000), P(0x10008), P(0x100000)
    # NULL required pointer
    assert lib.moe_route(c, None, good, None, good, good, ws, n, None) == L.MOE_ERR_INVALID_ARG
    # misaligned pointer
    assert lib.moe_route(c, odd, good, None, good, good, ws, n, None) == L.MOE_ERR_ALIGNMENT
    # workspace too small / misaligned
    assert lib.moe_route(c, good, good, None, good, good, ws, n - 256, None) == L.MOE_ERR_WORKSPACE
    assert lib.moe_route(c, good, good, None, good, good, P(0x100080), n, None) == L.MOE_ERR_ALIGNMENT
    assert lib.moe_permute(c, good, good, good, good, None, good, good, good, None, None, None,
                           None, ws, n, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_ffn(c, good, good, good, good, None, None, good, None, None, None, None,
                              ws, n, None) == L.MOE_ERR_INVALID_ARG
    # shared experts requested without their weights
    assert lib.moe_expert_ffn(c, good, good, good, good, good, None, good, good, None, None, good,
                              ws, n, None) == L.MOE_ERR_INVALID_ARG
    # an fp8-expert layer needs its moe_fp8_t, with every scale the call reads
    c8 = _cfg(dtype="bf16", flags=L.MOE_FLAG_FP8_EXPERTS)
    cc8 = C.byref(c8.c())
    n8 = _ws(lib, c8)
    assert lib.moe_expert_ffn(cc8, good, good, good, good, good, None, good, None, None, None,
                              None, ws, n8, None) == L.MOE_ERR_INVALID_ARG
    part = L.moe_fp8_t(w1_scale=0x10000, w3_scale=0x10000, w2_scale=0x10000, x_scale=0x10000)
    assert lib.moe_expert_ffn(cc8, good, good, good, good, good, C.byref(part), good, None, None,
                              None, None, ws, n8, None) == L.MOE_ERR_INVALID_ARG   # no h_scale
    assert lib.moe_permute(cc8, good, good, good, good, None, good, good, good, good, None, good,
                           C.byref(L.moe_fp8_t()), ws, n8, None) == L.MOE_ERR_INVALID_ARG
    w8 = L.moe_weights_t(w_router=0x10000, w_down=0x10000, rms_gamma=0x10000, w1=0x10000,
                         w3=0x10000, w2=0x10000, w1_s=0x10000, w3_s=0x10000, w2_s=0x10000,
                         w_up=0x10000)
    assert lib.moe_forward(cc8, C.byref(w8), good, good, ws, n8, None, None) == \
        L.MOE_ERR_INVALID_ARG
    cf8 = _cfg(flags=L.MOE_FLAG_FP8_EXPERTS)          # fp32 layer
    assert lib.moe_workspace_size(C.byref(cf8.c()), C.byref(C.c_size_t())) == L.MOE_ERR_UNSUPPORTED
    cs8 = _cfg(dtype="bf16", flags=L.MOE_FLAG_FP8_EXPERTS | L.MOE_FLAG_SIMT)
    assert lib.moe_workspace_size(C.byref(cs8.c()), C.byref(C.c_size_t())) == L.MOE_ERR_UNSUPPORTED
    c8w = _cfg(dtype="bf16", d_latent=64, flags=L.MOE_FLAG_FP8_EXPERTS)   # widths not /128
    assert lib.moe_workspace_size(C.byref(c8w.c()), C.byref(C.c_size_t())) == L.MOE_ERR_ALIGNMENT
    assert lib.moe_combine(c, good, good, None, None, None, None, good, ws, n, None) == \
        L.MOE_ERR_INVALID_ARG
    w = L.moe_weights_t(w_router=0x10000, w_down=0x10000, rms_gamma=0x10000, w1=0x10000,
                        w3=0x10000, w2=0x10000, w1_s=0x10000, w3_s=0x10000, w2_s=None,
                        w_up=0x10000)
    assert lib.moe_forward(c, C.byref(w), good, good, ws, n, None, None) == L.MOE_ERR_INVALID_ARG
    cfg2 = _cfg(pool_rows=100)                      # fewer pool rows than T * k
    assert lib.moe_forward(C.byref(cfg2.c()), C.byref(w), good, good, ws, n, None, None) == \
        L.MOE_ERR_INVALID_ARG
    assert lib.moe_get_device_status(None, 256, None, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_device_timeout(ws, 256, 0, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_device_timeout(ws, 256, 20000, None) == L.MOE_ERR_INVALID_ARG
    # a bf16 router needs a 16-byte row pitch of W_r (E a multiple of 8); the expert calls do not
    c12 = _cfg(dtype="bf16", n_experts=12)
    n12 = _ws(lib, c12)
    assert lib.moe_route(C.byref(c12.c()), good, good, None, good, good, ws, n12, None) == \
        L.MOE_ERR_ALIGNMENT


def test_binding_refuses_missing_library(tmp_path):
    from sparse_expert_router_gb300 import _lib
    saved = _lib._lib
    _lib._lib = None
    try:
        with pytest.raises(RuntimeError, match="missing"):
            _lib.load(str(tmp_path / "nope.so"))
    finally:
        _lib._lib = saved


def test_last_cuda_error_starts_clear(lib):
    name = C.c_char_p()
    assert lib.moe_last_cuda_error(C.byref(name)) == 0
    assert name.value == b"cudaSuccess"
    assert lib.moe_last_cuda_error(None) == 0


def test_backward_argument_errors(lib):
    from sparse_expert_router_gb300 import _lib as L
    P = lambda v: C.c_void_p(v)
    good, ws = P(0x10000), P(0x100000)
    cfg = _cfg(dtype="bf16", d_latent=128, d_ff=128)
    c = C.byref(cfg.c())
    n = C.c_size_t()
    assert lib.moe_backward_workspace_size(c, C.byref(n)) == L.MOE_OK and n.value > 0
    args = [good] * 10
    assert lib.moe_expert_ffn_backward(c, *args[:9], None, ws, n.value, None) == \
        L.MOE_ERR_INVALID_ARG                                          # dw2 missing
    assert lib.moe_expert_ffn_backward(c, *args, ws, n.value - 256, None) == L.MOE_ERR_WORKSPACE
    f32 = _cfg(d_latent=128, d_ff=128)                                 # fp32 layer
    assert lib.moe_expert_ffn_backward(C.byref(f32.c()), *args, ws, n.value, None) == \
        L.MOE_ERR_UNSUPPORTED
    odd = _cfg(dtype="bf16", d_latent=128, d_ff=64)                    # width not /128
    assert lib.moe_expert_ffn_backward(C.byref(odd.c()), *args, ws, n.value, None) == \
        L.MOE_ERR_ALIGNMENT


def test_layer_backward_argument_errors(lib):
    from sparse_expert_router_gb300 import _lib as L
    P = lambda v: C.c_void_p(v)
    good, ws = P(0x10000), P(0x100000)
    cfg = _cfg(dtype="bf16", d_model=256, d_latent=128, d_ff=128, n_experts=64, n_shared=1,
               d_ff_shared=128)
    c = C.byref(cfg.c())
    n = C.c_size_t()
    assert lib.moe_layer_backward_workspace_size(c, C.byref(n)) == L.MOE_OK
    fw = _ws(lib, cfg)
    w = L.moe_weights_t(**{f: 0x10000 for f in ("w_router", "w_down", "rms_gamma", "w1", "w3",
                                                "w2", "w1_s", "w3_s", "w2_s", "w_up")})
    grads = L.moe_grads_t(**{f: 0x10000 for f in L.GRAD_NAMES})
    ok_args = (C.byref(w), good, good, good, C.byref(grads), P(0x200000), fw, ws, n.value, None)
    none_g = L.moe_grads_t(**{f: 0x10000 for f in L.GRAD_NAMES if f != "dw_up"})
    assert lib.moe_backward(c, C.byref(w), good, good, good, C.byref(none_g), P(0x200000), fw,
                            ws, n.value, None) == L.MOE_ERR_INVALID_ARG        # dw_up missing
    assert lib.moe_backward(c, C.byref(w), good, good, good, C.byref(grads), P(0x200000), fw - 256,
                            ws, n.value, None) == L.MOE_ERR_WORKSPACE         # forward workspace
    assert lib.moe_backward(c, *ok_args[:-3], ws, n.value - 256, None) == L.MOE_ERR_WORKSPACE
    odd = _cfg(dtype="bf16", d_model=256, d_latent=128, d_ff=128, n_experts=48, n_shared=1,
               d_ff_shared=128)                                                # E not /64
    assert lib.moe_backward(C.byref(odd.c()), *ok_args) == L.MOE_ERR_UNSUPPORTED
    f32 = _cfg(d_model=256, d_latent=128, d_ff=128, n_experts=64)
    assert lib.moe_backward(C.byref(f32.c()), *ok_args) == L.MOE_ERR_UNSUPPORTED


def test_workspace_regions(lib):
    """The intermediates' offsets lie inside the workspace, 256-byte aligned, each region large
    enough for its tensor and none overlapping the next."""
    import sparse_expert_router_gb300 as m
    from sparse_expert_router_gb300 import _lib as L
    cfg = _cfg(dtype="bf16", T=300, pool_rows=0)
    r = m.workspace_regions(cfg)
    total = _ws(lib, cfg)
    T, Lt, F, k, E = 300, 128, 128, 2, 16
    sizes = {"z": T * Lt * 4, "x_perm": T * k * Lt * 2, "hidden": T * k * F * 2,
             "y_perm": T * k * Lt * 2, "a_shared": T * 256 * 2, "combined": T * Lt * 2,
             "perm": T * k * 4, "expert_offsets": (E + 1) * 4}
    spans = sorted((r[n], r[n] + sizes[n], n) for n in sizes)
    for (lo, hi, n), nxt in zip(spans, spans[1:] + [(total, total, "end")]):
        assert lo % 256 == 0 and hi <= nxt[0], (n, lo, hi, nxt)
    assert lib.moe_workspace_regions(C.byref(cfg.c()), None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_regions(None, C.byref(L.moe_workspace_regions_t())) == \
        L.MOE_ERR_INVALID_ARG
