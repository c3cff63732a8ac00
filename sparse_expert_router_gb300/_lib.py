"""ctypes view of the C ABI declared in include/moe_gb300.h (argument marshalling only)."""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_ALIGNMENT = 4
MOE_ERR_CUDA = 5
MOE_ERR_BAD_ROUTING = 6
MOE_ERR_DEVICE_TIMEOUT = 7

MOE_BF16 = 0
MOE_F32 = 1
MOE_FLAG_PDL = 1 << 0
MOE_FLAG_SIMT = 1 << 1
MOE_FLAG_FP8_EXPERTS = 1 << 2
MOE_FORWARD_STAGES = 8

STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_ALIGNMENT", 5: "MOE_ERR_CUDA",
                6: "MOE_ERR_BAD_ROUTING", 7: "MOE_ERR_DEVICE_TIMEOUT"}


class moe_config_t(C.Structure):
    _fields_ = [("T", C.c_int64), ("d_model", C.c_int32), ("d_latent", C.c_int32),
                ("n_experts", C.c_int32), ("top_k", C.c_int32), ("d_ff", C.c_int32),
                ("n_shared", C.c_int32), ("d_ff_shared", C.c_int32),
                ("capacity_num", C.c_int32), ("capacity_den", C.c_int32),
                ("rms_eps", C.c_float), ("dtype", C.c_int32), ("flags", C.c_uint32),
                ("pool_rows", C.c_int64)]


class moe_fp8_t(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("w1_scale", "w3_scale", "w2_scale", "x_scale",
                                          "h_scale", "x_amax", "h_amax")]


class moe_weights_t(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("w_router", "b_router", "w_down", "rms_gamma", "w1", "w3",
                                          "w2", "w1_s", "w3_s", "w2_s", "w_up")] + \
               [("fp8", C.POINTER(moe_fp8_t))]


GRAD_NAMES = ("dw_router", "db_router", "dw_down", "drms_gamma", "dw1", "dw3", "dw2", "dw1_s",
              "dw3_s", "dw2_s", "dw_up")


class moe_grads_t(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in GRAD_NAMES]


class moe_forward_aux_t(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("topk_idx", "topk_gate", "expert_counts",
                                          "expert_offsets", "slot_of", "n_dropped",
                                          "stage_events", "token_mask")]


REGION_NAMES = ("z", "x_perm", "hidden", "y_perm", "a_shared", "combined", "perm",
                "expert_offsets")


class moe_workspace_regions_t(C.Structure):
    _fields_ = [(n, C.c_size_t) for n in REGION_NAMES]


class moe_device_report_t(C.Structure):
    _fields_ = [("status", C.c_int32), ("detail", C.c_int32), ("n_refined", C.c_int32),
                ("n_exact", C.c_int32)]


P = C.c_void_p
CFG = C.POINTER(moe_config_t)

# name -> (restype, argtypes); the same names as the C ABI
SIGNATURES = {
    "moe_abi_version": (C.c_int32, []),
    "moe_status_string": (C.c_char_p, [C.c_int]),
    "moe_last_cuda_error": (C.c_int32, [C.POINTER(C.c_char_p)]),
    "moe_workspace_size": (C.c_int, [CFG, C.POINTER(C.c_size_t)]),
    "moe_workspace_regions": (C.c_int, [CFG, C.POINTER(moe_workspace_regions_t)]),
    "moe_route": (C.c_int, [CFG, P, P, P, P, P, P, C.c_size_t, P]),
    "moe_permute": (C.c_int, [CFG, P, P, P, P, P, P, P, P, P, P, P, C.POINTER(moe_fp8_t), P,
                              C.c_size_t, P]),
    "moe_expert_ffn": (C.c_int, [CFG, P, P, P, P, P, C.POINTER(moe_fp8_t), P, P, P, P, P, P,
                                 C.c_size_t, P]),
    "moe_combine": (C.c_int, [CFG, P, P, P, P, P, P, P, P, C.c_size_t, P]),
    "moe_backward_workspace_size": (C.c_int, [CFG, C.POINTER(C.c_size_t)]),
    "moe_layer_backward_workspace_size": (C.c_int, [CFG, C.POINTER(C.c_size_t)]),
    "moe_backward": (C.c_int, [CFG, C.POINTER(moe_weights_t), P, P, P, C.POINTER(moe_grads_t), P,
                               C.c_size_t, P, C.c_size_t, P]),
    "moe_expert_ffn_backward": (C.c_int, [CFG, P, P, P, P, P, P, P, P, P, P, P, C.c_size_t, P]),
    "moe_forward": (C.c_int, [CFG, C.POINTER(moe_weights_t), P, P, P, C.c_size_t, P,
                              C.POINTER(moe_forward_aux_t)]),
    "moe_forward_pipelined": (C.c_int, [CFG, C.POINTER(moe_weights_t), C.c_int32,
                                        C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), P, P, P,
                                        C.c_size_t, P, P, P]),
    "moe_get_device_status": (C.c_int, [P, C.c_size_t, P, C.POINTER(moe_device_report_t)]),
    "moe_clear_device_status": (C.c_int, [P, C.c_size_t, P]),
    "moe_route_noalloc": (C.c_int, [CFG, P, P, P, P, P, P, P]),
    "moe_selftest_device_timeout": (C.c_int, [P, C.c_size_t, C.c_uint32, P]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load the CUDA library. Raises if it has not been built: there is no fallback path."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m sparse_expert_router_gb300.build` "
            "(the routed-MoE layer runs only in its CUDA kernels)")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
