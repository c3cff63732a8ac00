"""GB300-native routed mixture-of-experts forward layer.

A thin Python binding over the C ABI of ``libmoe_gb300.so`` (include/moe_gb300.h): every
function here marshals torch tensors into pointers and sizes and calls the C entry point of
the same name; every step of the layer runs in the library's CUDA kernels. PyTorch supplies
device memory and streams only.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from typing import Dict, Optional, Sequence

import torch

from . import _lib
from ._lib import (GRAD_NAMES, MOE_BF16, MOE_F32, MOE_FLAG_FP8_EXPERTS, MOE_FLAG_PDL,
                   MOE_FLAG_SIMT, MOE_FORWARD_STAGES, moe_config_t, moe_device_report_t,
                   moe_forward_aux_t, moe_fp8_t, moe_grads_t, moe_weights_t)

__all__ = ["MoEError", "LayerConfig", "load", "workspace_size", "alloc_workspace", "moe_route",
           "moe_permute", "moe_expert_ffn", "moe_combine", "moe_forward",
           "backward_workspace_size", "alloc_backward_workspace", "moe_expert_ffn_backward",
           "layer_backward_workspace_size", "alloc_layer_backward_workspace", "moe_backward",
           "moe_forward_pipelined",
           "GRAD_NAMES",
           "moe_get_device_status", "moe_clear_device_status", "moe_route_noalloc",
           "moe_selftest_device_timeout",
           "MOE_FLAG_PDL", "MOE_FLAG_SIMT", "MOE_FLAG_FP8_EXPERTS",
           "MOE_FORWARD_STAGES", "WEIGHT_NAMES", "FP8_NAMES"]

WEIGHT_NAMES = ("w_router", "b_router", "w_down", "rms_gamma", "w1", "w3", "w2", "w1_s", "w3_s",
                "w2_s", "w_up")
# moe_fp8_t: weight column scales, activation multipliers (inputs) and amax (outputs)
FP8_NAMES = ("w1_scale", "w3_scale", "w2_scale", "x_scale", "h_scale", "x_amax", "h_amax")


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = f"{fn} returned {_lib.STATUS_NAMES.get(status, status)}"
        if status == 5:   # MOE_ERR_CUDA: name the CUDA error behind it
            name = C.c_char_p()
            code = load().moe_last_cuda_error(C.byref(name))
            msg += f" ({name.value.decode() if name.value else '?'}, {code})"
        super().__init__(msg)


@dataclass
class LayerConfig:
    T: int
    d_model: int
    d_latent: int
    n_experts: int
    top_k: int
    d_ff: int
    n_shared: int
    d_ff_shared: int
    dtype: str = "bf16"            # "bf16" or "f32"
    capacity: Optional[Sequence[int]] = None   # (num, den) or None
    rms_eps: float = 1e-6
    flags: int = 0
    pool_rows: int = 0

    @classmethod
    def from_shape(cls, shape, **kw) -> "LayerConfig":
        if getattr(shape, "expert_dtype", "bf16") == "fp8":
            kw["flags"] = kw.get("flags", 0) | MOE_FLAG_FP8_EXPERTS
        return cls(T=shape.T, d_model=shape.d_model, d_latent=shape.d_latent,
                   n_experts=shape.n_experts, top_k=shape.top_k, d_ff=shape.d_ff,
                   n_shared=shape.n_shared, d_ff_shared=shape.d_ff_shared, dtype=shape.dtype,
                   capacity=shape.capacity, rms_eps=shape.rms_eps, **kw)

    def c(self) -> moe_config_t:
        num, den = (self.capacity if self.capacity else (0, 1))
        return moe_config_t(T=self.T, d_model=self.d_model, d_latent=self.d_latent,
                            n_experts=self.n_experts, top_k=self.top_k, d_ff=self.d_ff,
                            n_shared=self.n_shared, d_ff_shared=self.d_ff_shared,
                            capacity_num=num, capacity_den=den, rms_eps=self.rms_eps,
                            dtype=MOE_BF16 if self.dtype == "bf16" else MOE_F32,
                            flags=self.flags, pool_rows=self.pool_rows)


def load():
    return _lib.load()


def _p(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _fp8(fp8: Optional[Dict[str, torch.Tensor]]):
    """A moe_fp8_t from a dict of device tensors named as its fields (missing ones NULL)."""
    if fp8 is None:
        return None
    return C.pointer(moe_fp8_t(**{n: (fp8[n].data_ptr() if fp8.get(n) is not None else None)
                                  for n in FP8_NAMES}))


def _check(fn: str, status: int):
    if status != 0:
        raise MoEError(fn, status)


def workspace_size(cfg: LayerConfig) -> int:
    n = C.c_size_t(0)
    _check("moe_workspace_size", load().moe_workspace_size(C.byref(cfg.c()), C.byref(n)))
    return n.value


def workspace_regions(cfg: LayerConfig) -> Dict[str, int]:
    """Byte offsets in the workspace of the intermediates moe_forward leaves there."""
    r = _lib.moe_workspace_regions_t()
    _check("moe_workspace_regions", load().moe_workspace_regions(C.byref(cfg.c()), C.byref(r)))
    return {n: int(getattr(r, n)) for n in _lib.REGION_NAMES}


def workspace_view(ws: torch.Tensor, cfg: LayerConfig, name: str, dtype: torch.dtype,
                   shape) -> torch.Tensor:
    """A tensor view of one region of the workspace (see workspace_regions)."""
    off = workspace_regions(cfg)[name]
    n = 1
    for s in shape:
        n *= int(s)
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype).view(*shape)


def alloc_workspace(cfg: LayerConfig, device="cuda") -> torch.Tensor:
    """A caller-owned, zero-filled workspace of the right size (torch's allocator aligns it to
    256 bytes); zero fill clears the device report it starts with."""
    return torch.zeros(workspace_size(cfg), dtype=torch.uint8, device=device)


def moe_route(cfg, x, w_router, b_router, topk_idx, topk_gate, ws, stream=None):
    _check("moe_route", load().moe_route(C.byref(cfg.c()), _p(x), _p(w_router), _p(b_router),
                                          _p(topk_idx), _p(topk_gate), _p(ws), ws.numel(),
                                          _stream(stream)))


def moe_permute(cfg, x, w_down, rms_gamma, topk_idx, expert_counts, expert_offsets, perm,
                slot_of, n_dropped, x_perm, ws, stream=None, fp8=None, token_mask=None):
    """``fp8``: dict of moe_fp8_t fields (x_scale, optional x_amax) for an fp8-expert layer.
    ``token_mask``: [T] uint8, 0 for attention-mask padding (not dispatched), or None."""
    _check("moe_permute", load().moe_permute(
        C.byref(cfg.c()), _p(x), _p(w_down), _p(rms_gamma), _p(topk_idx), _p(token_mask),
        _p(expert_counts),
        _p(expert_offsets), _p(perm), _p(slot_of), _p(n_dropped), _p(x_perm), _fp8(fp8), _p(ws),
        ws.numel(), _stream(stream)))


def moe_expert_ffn(cfg, x_perm, expert_offsets, w1, w3, w2, y_perm, x=None, w1_s=None,
                   w3_s=None, a_shared=None, ws=None, stream=None, fp8=None):
    """``fp8``: dict of moe_fp8_t fields for an fp8-expert layer (scales, optional h_amax)."""
    _check("moe_expert_ffn", load().moe_expert_ffn(
        C.byref(cfg.c()), _p(x_perm), _p(expert_offsets), _p(w1), _p(w3), _p(w2), _fp8(fp8),
        _p(y_perm), _p(x), _p(w1_s), _p(w3_s), _p(a_shared), _p(ws), ws.numel(),
        _stream(stream)))


def backward_workspace_size(cfg: LayerConfig) -> int:
    n = C.c_size_t(0)
    _check("moe_backward_workspace_size",
           load().moe_backward_workspace_size(C.byref(cfg.c()), C.byref(n)))
    return n.value


def alloc_backward_workspace(cfg: LayerConfig, device="cuda") -> torch.Tensor:
    """Zero-filled workspace of moe_expert_ffn_backward."""
    return torch.zeros(backward_workspace_size(cfg), dtype=torch.uint8, device=device)


def moe_expert_ffn_backward(cfg, x_perm, expert_offsets, w1, w3, w2, dy_perm, dx_perm, dw1, dw3,
                            dw2, ws, stream=None):
    _check("moe_expert_ffn_backward", load().moe_expert_ffn_backward(
        C.byref(cfg.c()), _p(x_perm), _p(expert_offsets), _p(w1), _p(w3), _p(w2), _p(dy_perm),
        _p(dx_perm), _p(dw1), _p(dw3), _p(dw2), _p(ws), ws.numel(), _stream(stream)))


def layer_backward_workspace_size(cfg: LayerConfig) -> int:
    n = C.c_size_t(0)
    _check("moe_layer_backward_workspace_size",
           load().moe_layer_backward_workspace_size(C.byref(cfg.c()), C.byref(n)))
    return n.value


def alloc_layer_backward_workspace(cfg: LayerConfig, device="cuda") -> torch.Tensor:
    """Zero-filled workspace of moe_backward."""
    return torch.zeros(layer_backward_workspace_size(cfg), dtype=torch.uint8, device=device)


def moe_backward(cfg, weights: Dict[str, torch.Tensor], x, dy, dx, grads: Dict[str, torch.Tensor],
                 fwd_ws, ws, stream=None):
    """dx and the weight gradients (``grads`` maps GRAD_NAMES to device tensors; db_router and
    drms_gamma may be missing) of the layer whose moe_forward used ``fwd_ws`` on x."""
    w = moe_weights_t(**{n: (weights[n].data_ptr() if weights.get(n) is not None else None)
                         for n in WEIGHT_NAMES})
    g = moe_grads_t(**{n: (grads[n].data_ptr() if grads.get(n) is not None else None)
                       for n in GRAD_NAMES})
    _check("moe_backward", load().moe_backward(
        C.byref(cfg.c()), C.byref(w), _p(x), _p(dy), _p(dx), C.byref(g), _p(fwd_ws),
        fwd_ws.numel(), _p(ws), ws.numel(), _stream(stream)))


def moe_combine(cfg, y_perm, slot_of, topk_gate, out, ws, a_shared=None, w_up=None, w2_s=None,
                stream=None):
    _check("moe_combine", load().moe_combine(
        C.byref(cfg.c()), _p(y_perm), _p(slot_of), _p(topk_gate), _p(a_shared), _p(w_up),
        _p(w2_s), _p(out), _p(ws), ws.numel(), _stream(stream)))


def moe_forward(cfg, weights: Dict[str, torch.Tensor], x, y, ws, stream=None,
                aux: Optional[Dict[str, object]] = None):
    """y = layer(x). ``aux`` may map topk_idx / topk_gate / expert_counts / expert_offsets /
    slot_of / n_dropped to device tensors, token_mask to a [T] uint8 input (0 = padding, not
    dispatched), and stage_events to MOE_FORWARD_STAGES + 1
    torch.cuda.Event objects (created with enable_timing=True). For an fp8-expert layer
    ``weights`` also holds w1_scale, w3_scale, w2_scale, x_scale and h_scale, and ``aux`` may
    map x_amax / h_amax to [1] fp32 device tensors."""
    w = moe_weights_t(**{n: (weights[n].data_ptr() if weights.get(n) is not None else None)
                         for n in WEIGHT_NAMES})
    if cfg.flags & MOE_FLAG_FP8_EXPERTS:
        f8 = {n: weights.get(n) for n in FP8_NAMES[:5]}
        f8.update({n: (aux or {}).get(n) for n in FP8_NAMES[5:]})
        fp8_ref = _fp8(f8)
        w.fp8 = fp8_ref
    a = None
    keep = None
    if aux:
        fields = {n: (aux[n].data_ptr() if aux.get(n) is not None else None)
                  for n in ("topk_idx", "topk_gate", "expert_counts", "expert_offsets",
                            "slot_of", "n_dropped", "token_mask")}
        if aux.get("stage_events") is not None:
            evs = aux["stage_events"]
            keep = (C.c_void_p * len(evs))(*[e.cuda_event for e in evs])
            fields["stage_events"] = C.cast(keep, C.c_void_p).value
        a = moe_forward_aux_t(**fields)
    _check("moe_forward", load().moe_forward(C.byref(cfg.c()), C.byref(w), _p(x), _p(y), _p(ws),
                                             ws.numel(), _stream(stream),
                                             C.byref(a) if a is not None else None))
    del keep


def moe_forward_pipelined(cfg, weights: Dict[str, torch.Tensor], x_hosts, y_hosts, x_stage,
                          y_stage, ws, stream, h2d_stream, d2h_stream):
    """moe_forward over host batches x_hosts[i] -> y_hosts[i] (pinned CPU tensors), copies
    overlapped with the forwards on two more streams; x_stage / y_stage: [2, T, d] device."""
    w = moe_weights_t(**{n: (weights[n].data_ptr() if weights.get(n) is not None else None)
                         for n in WEIGHT_NAMES})
    keep = None
    if cfg.flags & MOE_FLAG_FP8_EXPERTS:
        keep = _fp8({n: weights.get(n) for n in FP8_NAMES[:5]})
        w.fp8 = keep
    n = len(x_hosts)
    xs = (C.c_void_p * n)(*[t.data_ptr() for t in x_hosts])
    ys = (C.c_void_p * n)(*[t.data_ptr() for t in y_hosts])
    _check("moe_forward_pipelined", load().moe_forward_pipelined(
        C.byref(cfg.c()), C.byref(w), n, xs, ys, _p(x_stage), _p(y_stage), _p(ws), ws.numel(),
        _stream(stream), _stream(h2d_stream), _stream(d2h_stream)))
    del keep


def moe_get_device_status(ws, stream=None) -> Dict[str, int]:
    r = moe_device_report_t()
    _check("moe_get_device_status",
           load().moe_get_device_status(_p(ws), ws.numel(), _stream(stream), C.byref(r)))
    return {"status": r.status, "detail": r.detail, "n_refined": r.n_refined,
            "n_exact": r.n_exact}


def moe_selftest_device_timeout(ws, limit_ms=200, stream=None):
    """Enqueue a bounded wait that nothing satisfies; it records MOE_ERR_DEVICE_TIMEOUT."""
    _check("moe_selftest_device_timeout",
           load().moe_selftest_device_timeout(_p(ws), ws.numel(), int(limit_ms), _stream(stream)))


def moe_clear_device_status(ws, stream=None):
    _check("moe_clear_device_status",
           load().moe_clear_device_status(_p(ws), ws.numel(), _stream(stream)))


def moe_route_noalloc(cfg, x, w_router, b_router, topk_idx, topk_gate, device_report=None,
                      stream=None):
    """moe_route for callers that cannot allocate device memory: no workspace argument; the
    library's fixed 32 MiB scratch array is used instead (see include/moe_gb300.h)."""
    _check("moe_route_noalloc", load().moe_route_noalloc(
        C.byref(cfg.c()), _p(x), _p(w_router), _p(b_router), _p(topk_idx), _p(topk_gate),
        _p(device_report), _stream(stream)))
