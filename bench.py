"""Benchmark of the routed-MoE forward layer on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step is one forward of the whole layer (router, top-k, dispatch, grouped expert GEMMs,
shared experts, combine, up-projection) over one batch of synthetic tokens of the workload
(default: the 535B-shaped layer, T = 8,192 tokens). Prints one JSON line on rank 0.

For N > 1 (torchrun, one process per GPU) every rank runs its own replica of the layer on its
own batch (token sharding, no collective on the data path); the barrier and the max over ranks
are used for timing only ("replicas only" scaling, reported as weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from moe_workloads import SHAPES, make_layer_inputs  # noqa: E402

STAGES = ["prep", "front_gemm", "router_select", "dispatch", "expert_gemm1", "expert_gemm2",
          "combine", "back_gemm"]
def launches_per_forward(shape, simt: bool) -> int:
    """This library's kernel launches in one moe_forward: the device-report reset, router
    preparation (2), the front GEMMs (one tensor-core launch; two from 0.5 TFLOP of front GEMMs
    up, when the down-projection and shared experts run as CTA pairs beside the router's launch;
    or one CUDA-core launch per problem), the router (3), dispatch (3), the expert GEMMs (2), then
    the combine and the back GEMM (one launch when the combine runs inside the tensor-core back
    GEMM)."""
    tc = shape.dtype == "bf16" and not simt
    pairs = os.environ.get("MOE_TC_PAIR", "1") in ("1", "dual") if shape.n_shared == 0 else \
        os.environ.get("MOE_TC_PAIR", "1") == "1"
    env_split = os.environ.get("MOE_FRONT_SPLIT")
    front_flops = 2.0 * shape.T * shape.d_model * (shape.n_experts + shape.d_latent
                                                    + 2 * shape.n_shared * shape.d_ff_shared)
    split = (tc and pairs and (front_flops >= 0.5e12 if env_split is None else env_split != "0")
             and shape.d_latent % 512 == 0
             and (shape.n_shared == 0 or shape.d_ff_shared % 256 == 0))
    front = (2 if split else 1) if tc else 2 + (1 if shape.n_shared > 0 else 0)
    env = os.environ.get("MOE_FUSED_COMBINE")
    rows_bytes = shape.T * shape.top_k * shape.d_latent * 2
    fused = tc and shape.n_shared > 0 and (rows_bytes <= (96 << 20) if env is None else env != "0")
    return 1 + 2 + front + 3 + 3 + 2 + (1 if fused else 2)
METRIC = "MoE-layer tokens/s"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_burst": p["bf16_tflops"],
                "bf16_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_burst": 1900.0, "bf16_sustained": 1700.0,
                "source": "fallback"}


# ncu summaries with per-launch DRAM traffic, each with the sources its kernels are compiled from:
# a change to any of them voids that summary's counters
PROFILE_SUMMARIES = (
    (os.path.join(ROOT, "profiles", "tc_gemm_grouped_l535b_e64_t1368.md"),
     ("gemm_tc.cu", "tc_ptx.cuh", "common.cuh", "gemm.h")),
    (os.path.join(ROOT, "profiles", "memory_kernels_l535b_f128_t8192.md"),
     ("dispatch.cu", "router.cu", "common.cuh")),
)


def profiled_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu summaries, or None
    when there is none or a source of the kernel changed since the counters were taken."""
    import hashlib
    for path, sources in PROFILE_SUMMARIES:
        try:
            text = open(path).read()
            shas = {f: hashlib.sha256(open(os.path.join(ROOT, "sparse_expert_router_gb300", "csrc",
                                                        f), "rb").read()).hexdigest()[:16]
                    for f in sources}
        except OSError:
            continue
        lines = [ln.split() for ln in text.splitlines()]
        if any(["source_sha256_prefix", f, sha] not in lines for f, sha in shas.items()):
            continue
        for parts in lines:
            if len(parts) == 4 and parts[0] == "traffic_per_launch" and parts[1] == workload \
                    and parts[2] == kernel:
                return float(parts[3])
    return None


def max_over_ranks(x: float, device) -> float:
    """Max of a per-rank float over the process group (the value itself on one process)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def algorithmic(shape, kept):
    """Algorithmic flops and bytes per stage of one forward, given the rows each expert keeps
    after the capacity clamp (`kept`, the differences of the group offsets): bf16 storage,
    except that an fp8-expert layer keeps its expert banks (plus one fp32 scale per output
    column), grouped rows and hidden in E4M3 (one byte). "tc_peak" names the tensor-core rate a
    stage runs at."""
    T, d, L, E, k = shape.T, shape.d_model, shape.d_latent, shape.n_experts, shape.top_k
    F, SF = shape.d_ff, shape.n_shared * shape.d_ff_shared
    es = 4 if shape.dtype == "f32" else 2
    fp8 = getattr(shape, "expert_dtype", "bf16") == "fp8"
    wb = 1 if fp8 else es                              # bytes per expert-bank weight
    ab = 1 if fp8 else es                              # bytes per grouped-row / hidden value
    xp = "fp8" if fp8 else "bf16"
    R = int(sum(kept))
    active = sum(1 for c in kept if c > 0)
    fl = shape.flops()
    fl["expert_up"] = 2.0 * R * L * 2 * F
    fl["expert_down"] = 2.0 * R * F * L
    return {
        "front_gemm": {"flops": fl["router"] + fl["down"] + fl["shared_up"],
                       "bytes": es * (T * d + d * E + d * L + 2 * d * SF) + 4 * T * E + 4 * T * L
                       + es * T * SF},
        "router_select": {"flops": 0.0, "bytes": 4 * T * E + es * T * d + 8 * T * k},
        "dispatch": {"flops": 0.0, "bytes": 4 * T * L + ab * R * L + 4 * (3 * T * k + R)},
        "expert_gemm1": {"flops": fl["expert_up"], "tc_peak": xp,
                         "bytes": wb * 2 * active * L * F + ab * (R * L + R * F)
                         + (8 * active * F if fp8 else 0)},
        "expert_gemm2": {"flops": fl["expert_down"], "tc_peak": xp,
                         "bytes": wb * active * F * L + ab * R * F + es * R * L
                         + (4 * active * L if fp8 else 0)},
        "combine": {"flops": 0.0, "bytes": es * (R * L + T * L) + 8 * T * k},
        "back_gemm": {"flops": fl["back"],
                      "bytes": es * (T * L + T * SF + L * d + SF * d + T * d)},
    }


def weight_bytes(shape) -> int:
    """Bytes of every weight of the layer as stored."""
    d, L, E, F = shape.d_model, shape.d_latent, shape.n_experts, shape.d_ff
    SF = shape.n_shared * shape.d_ff_shared
    bank = 3 * E * L * F * (1 if shape.expert_dtype == "fp8" else 2)
    scales = 4 * E * (2 * F + L) if shape.expert_dtype == "fp8" else 0
    return bank + scales + 2 * (d * E + 2 * d * L + 3 * d * SF) + 4 * (E + L)


def f32_alu_peak(dev, clk) -> float:
    """Peak of the CUDA-core fp32 GEMMs (TFLOP/s), derived from unit counts and clock: every SM's
    128 fp32 lanes issuing one fused multiply-add (2 flops) a clock at the highest SM clock seen
    (2,070 MHz when none was sampled): ~80.5 TFLOP/s on 152 SMs."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = (clk or {}).get("sm_max_mhz") or 2070.0
    return sms * 128 * 2 * mhz * 1e6 / 1e12


def tc_peak(pk, stage, which="bf16_burst") -> float:
    """Tensor-core peak (TFLOP/s) of a stage: the measured bf16 rate (burst by default: the timed
    loops here last a fraction of a second; "bf16_sustained" for the seconds-long rate under the
    power cap), doubled for E4M3 operands (the nominal dense ratio 4.5 / 2.25 PFLOP/s)."""
    return pk[which] * (2.0 if stage.get("tc_peak") == "fp8" else 1.0)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = str(index)
        try:   # nvidia-smi numbers GPUs differently from CUDA when devices are masked
            uuid = str(torch.cuda.get_device_properties(index).uuid)
            if uuid:
                self.index = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except (AttributeError, RuntimeError):
            pass
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", self.index], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args, shape):
    """The fp64 CPU oracle timed on the host cores, each step a bounded sample of the workload."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from oracle import moe_oracle
    gen = "cuda" if torch.cuda.is_available() else "cpu"
    inp = {k: v.cpu() for k, v in make_layer_inputs(shape, gen, T=args.ref_tokens).items()}
    for _ in range(args.warmup if args.warmup <= 1 else 1):
        moe_oracle.forward(inp, top_k=shape.top_k, rms_eps=shape.rms_eps,
                           capacity_factor=shape.capacity)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        moe_oracle.forward(inp, top_k=shape.top_k, rms_eps=shape.rms_eps,
                           capacity_factor=shape.capacity)
    dt = time.perf_counter() - t0
    v = args.ref_tokens * args.steps / dt
    sample = f"{args.ref_tokens} tokens of {shape.name} per step (full weights)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) activations, N(0,1/fan_in) weights)",
        "config": forward_config(shape, args, world),
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": torch.get_num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def cpu_baseline(shape, n_tokens, inp_gpu):
    """The oracle as it stands on a bounded token sample, with the workload's weights on the host."""
    from oracle import moe_oracle
    host = {k: v.cpu() for k, v in inp_gpu.items()}
    host["x"] = host["x"][:n_tokens].clone()
    t0 = time.perf_counter()
    moe_oracle.forward(host, top_k=shape.top_k, rms_eps=shape.rms_eps,
                       capacity_factor=shape.capacity)
    dt = time.perf_counter() - t0
    return {"value": n_tokens / dt, "unit": "tokens/s", "cores": torch.get_num_threads(),
            "kind": "oracle", "seconds": dt,
            "sample": f"the first {n_tokens} tokens of {shape.name} as one batch "
                      f"(routing, dispatch, every expert MLP, combine, shared, up-projection)"}


def run_expert_backward(args, shape):
    """Backward of the routed expert MLP on the workload's own routing: moe_route and
    moe_permute give the grouped rows and offsets, dy_perm is seeded N(0, 1) bf16, and each step
    is one moe_expert_ffn_backward call (recompute, dA, dX, dW2, dW1 and dW3). One GPU."""
    import sparse_expert_router_gb300 as m
    m.load()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    flags = 0 if args.no_pdl else m.MOE_FLAG_PDL
    cfg = m.LayerConfig.from_shape(shape, flags=flags)
    T, k, E, L, F = shape.T, shape.top_k, shape.n_experts, shape.d_latent, shape.d_ff
    inp = make_layer_inputs(shape, dev)
    ws = m.alloc_workspace(cfg, dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    gate = torch.empty((T, k), dtype=torch.float32, device=dev)
    m.moe_route(cfg, inp["x"], inp["w_router"], inp["b_router"], idx, gate, ws)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    slot = torch.empty((T, k), dtype=torch.int32, device=dev)
    ndrop = torch.empty(1, dtype=torch.int32, device=dev)
    xp = torch.empty((T * k, L), dtype=torch.bfloat16, device=dev)
    m.moe_permute(cfg, inp["x"], inp["w_down"], inp["rms_gamma"], idx, counts, offs, perm, slot,
                  ndrop, xp, ws)
    g = torch.Generator(device=dev).manual_seed(7)
    dy = torch.randn((T * k, L), generator=g, device=dev).to(torch.bfloat16)
    dx = torch.empty_like(xp)
    dw1, dw3, dw2 = (torch.empty_like(inp[n]) for n in ("w1", "w3", "w2"))
    bws = m.alloc_backward_workspace(cfg, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream(dev)

    def step():
        m.moe_expert_ffn_backward(cfg, xp, offs, inp["w1"], inp["w3"], inp["w2"], dy, dx, dw1,
                                  dw3, dw2, bws, stream=st)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    clk = ClockSampler(0)
    clk.start()
    ms = 0.0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(args.steps):
        flush.zero_()
        a.record(st)
        step()
        b.record(st)
        b.synchronize()
        ms += a.elapsed_time(b)
    clocks = clk.stop()
    ms /= args.steps
    rep = m.moe_get_device_status(bws)
    R = int(offs[-1].item())
    active = int((counts > 0).sum().item())
    flops = 16.0 * R * L * F          # recompute 4RLF, dA 2RFL, dX 4RFL, dW2 2RFL, dW1+dW3 4RLF
    # bf16 bytes of this design's passes: W1 and W3 read twice and W2 once, the three weight
    # gradients written; rows: x read 3x, dy 2x, dx written; G, U, A and dG, dU written (5x),
    # then read (G, U by dA; A by dW2; dG, dU by dX and by dW1 / dW3: 7x)
    by = 2 * 5 * active * L * F + 2 * 3 * active * L * F + 2 * R * 6 * L + 2 * R * 12 * F
    pk = peaks()
    if by / (pk["hbm_gbs"] * 1e9) >= flops / (pk["bf16_burst"] * 1e12):
        ach = by / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / pk["hbm_gbs"], 4), "peak_source": pk["source"] + " (HBM copy)"}
    else:
        ach = flops / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": pk["bf16_burst"],
                "unit": "TFLOP/s", "frac": round(ach / pk["bf16_burst"], 4),
                "sustained_frac": round(ach / pk["bf16_sustained"], 4),
                "peak_source": pk["source"] + " (bf16 burst)"}
    roof["traffic"] = None
    print(json.dumps({
        "metric": "routed-expert MLP backward tokens/s", "value": round(T / (ms * 1e-3), 1),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic (the workload's routing of seeded inputs; dy_perm seeded N(0,1))",
        "config": {"workload": f"{shape.name}: T={T} E={E} k={k} L={L} F={F}", "rows": R,
                   "pdl": not args.no_pdl, "l2": "flushed between timed steps (256 MB write)"},
        "tflop_s": round(flops / (ms * 1e-3) / 1e12, 1),
        "roofline": roof, "gpu_launches": 7 * args.steps, "clocks": clocks, "device_report": rep}))


def run_layer_backward(args, shape):
    """The whole layer's backward (moe_backward) after one moe_forward on the workload; each
    step is one backward call with a seeded bf16 dy. One GPU."""
    import sparse_expert_router_gb300 as m
    m.load()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    cfg = m.LayerConfig.from_shape(shape, flags=0 if args.no_pdl else m.MOE_FLAG_PDL)
    T, d, L, E, F = shape.T, shape.d_model, shape.d_latent, shape.n_experts, shape.d_ff
    S, Fs = shape.n_shared, shape.d_ff_shared
    inp = make_layer_inputs(shape, dev)
    fws = m.alloc_workspace(cfg, dev)
    y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    counts = torch.zeros(E, dtype=torch.int32, device=dev)
    m.moe_forward(cfg, inp, inp["x"], y, fws, aux={"expert_counts": counts})
    g = torch.Generator(device=dev).manual_seed(7)
    dy = torch.randn((T, d), generator=g, device=dev).to(torch.bfloat16)
    dx = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    grads = {n: torch.empty_like(inp[n[1:]]) for n in m.GRAD_NAMES
             if n not in ("db_router", "drms_gamma")}
    grads["db_router"] = torch.empty(E, dtype=torch.float32, device=dev)
    grads["drms_gamma"] = torch.empty(L, dtype=torch.float32, device=dev)
    bws = m.alloc_layer_backward_workspace(cfg, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream(dev)

    def step():
        m.moe_backward(cfg, inp, inp["x"], dy, dx, grads, fws, bws, stream=st)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    clk = ClockSampler(0)
    clk.start()
    ms = 0.0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(args.steps):
        flush.zero_()
        a.record(st)
        step()
        b.record(st)
        b.synchronize()
        ms += a.elapsed_time(b)
    clocks = clk.stop()
    ms /= args.steps
    R = int(min(int(counts.sum()), T * shape.top_k))
    SF = S * Fs
    # flops: the experts' backward (16 R L F), the dense gradients: dc and dW_up (2 x 2TLd),
    # shared recompute (4 T d SF), shared dA and dW2s (2 x 2 T SF d), dx and dW for the
    # down-projection (2 x 2 T d L), for the shared gate/up (2 x 4 T d SF), router (2 x 2 T d E)
    flops = 16.0 * R * L * F + 2.0 * T * (2 * L * d + 4 * d * SF + 2 * SF * d + 2 * d * L
                                          + 4 * d * SF + 2 * d * E)
    pk = peaks()
    ach = flops / (ms * 1e-3) / 1e12
    print(json.dumps({
        "metric": "MoE-layer backward tokens/s", "value": round(T / (ms * 1e-3), 1),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic (seeded layer inputs, the forward's routing, dy seeded N(0,1))",
        "config": {"workload": f"{shape.name}: T={T} d={d} latent={L} E={E} "
                               f"k={shape.top_k} F={F} shared={S}x{Fs}",
                   "pdl": not args.no_pdl, "l2": "flushed between timed steps (256 MB write)"},
        "tflop_s": round(ach, 1),
        "roofline": {"bound": "tensor", "achieved": round(ach, 1), "peak": pk["bf16_burst"],
                     "unit": "TFLOP/s", "frac": round(ach / pk["bf16_burst"], 4),
                     "sustained_frac": round(ach / pk["bf16_sustained"], 4),
                     "traffic": None, "peak_source": pk["source"] + " (bf16 burst)"},
        "clocks": clocks, "device_report": m.moe_get_device_status(bws)}))


def run_slice(args):
    """One expert-parallel rank's slice of the 535B layer: 49,152 rows that arrive tagged with
    6 local experts (Dirichlet(0.5) shares) in a padded pool of 56,576, run through the grouped
    SwiGLU expert MLP (moe_expert_ffn) and the gate-weighted un-permute back to arrival order
    (moe_combine without an up-projection). One GPU; no routing, no shared experts."""
    import sparse_expert_router_gb300 as m
    from moe_workloads import SLICE_C5B, make_slice_inputs
    m.load()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    sh = SLICE_C5B
    cfg = m.LayerConfig(T=sh.rows, d_model=sh.d_latent, d_latent=sh.d_latent,
                        n_experts=sh.n_local, top_k=1, d_ff=sh.d_ff, n_shared=0, d_ff_shared=0,
                        dtype=sh.dtype, pool_rows=sh.pool_rows,
                        flags=0 if args.no_pdl else m.MOE_FLAG_PDL)
    inp = make_slice_inputs(sh, dev)
    ws = m.alloc_workspace(cfg, dev)
    y_perm = torch.empty((sh.pool_rows, sh.d_latent), dtype=torch.bfloat16, device=dev)
    out = torch.empty((sh.rows, sh.d_latent), dtype=torch.bfloat16, device=dev)
    slot, gate = inp["slot_of"].view(-1, 1), inp["gate"].view(-1, 1)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def step():
        ev[0].record(st)
        m.moe_expert_ffn(cfg, inp["pool"], inp["expert_offsets"], inp["w1"], inp["w3"],
                         inp["w2"], y_perm, ws=ws, stream=st)
        ev[1].record(st)
        m.moe_combine(cfg, y_perm, slot, gate, out, ws, stream=st)
        ev[2].record(st)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    clk = ClockSampler(0)
    clk.start()
    tot = ffn = comb = 0.0
    for _ in range(args.steps):
        flush.zero_()
        step()
        ev[2].synchronize()
        ffn += ev[0].elapsed_time(ev[1])
        comb += ev[1].elapsed_time(ev[2])
    clocks = clk.stop()
    ffn /= args.steps
    comb /= args.steps
    ms = ffn + comb
    R, L, F = sh.rows, sh.d_latent, sh.d_ff
    flops = 6.0 * R * L * F                 # gate, up (4RLF) and down (2RFL) projections
    pk = peaks()
    ach = flops / (ffn * 1e-3) / 1e12
    comb_bytes = 2 * (R * L + R * L) + 8 * R   # rows read, outputs written, gates and slots
    print(json.dumps({
        "metric": "expert-slice rows/s", "value": round(R / (ms * 1e-3), 1), "unit": "rows/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic (seeded rows, Dirichlet(0.5) expert shares, U(0,1] gates)",
        "config": {"workload": f"{sh.name}: rows={R} pool={sh.pool_rows} L={L} F={F} "
                               f"local experts={sh.n_local}", "pdl": not args.no_pdl,
                   "l2": "flushed between timed steps (256 MB write)"},
        "stages": {"expert_ffn": {"ms": round(ffn, 4), "tflop_s": round(ach, 1)},
                   "combine": {"ms": round(comb, 4),
                               "gb_s": round(comb_bytes / (comb * 1e-3) / 1e9, 1)}},
        "roofline": {"bound": "tensor", "achieved": round(ach, 1), "peak": pk["bf16_burst"],
                     "unit": "TFLOP/s", "frac": round(ach / pk["bf16_burst"], 4),
                     "sustained_frac": round(ach / pk["bf16_sustained"], 4),
                     "kernel": "expert_ffn", "traffic": None,
                     "peak_source": pk["source"] + " (bf16 burst)"},
        "gpu_launches": 4 * args.steps, "clocks": clocks,   # offsets check, 2 GEMMs, combine
        "device_report": m.moe_get_device_status(ws),
        **({} if args.no_cpu_baseline else {"cpu_baseline": slice_cpu_baseline(inp, 1024)})}))


def slice_cpu_baseline(inp_gpu, n_rows):
    """The oracle's slice on a bounded sample of arrival positions (every expert's rows)."""
    from oracle import moe_oracle
    host = {k: v.cpu() for k, v in inp_gpu.items()}
    n = host["slot_of"].numel()
    pos = torch.linspace(0, n - 1, n_rows).round().long().tolist()
    t0 = time.perf_counter()
    moe_oracle.slice_rows(host, pos)
    dt = time.perf_counter() - t0
    return {"value": n_rows / dt, "unit": "rows/s", "cores": torch.get_num_threads(),
            "kind": "oracle", "seconds": dt,
            "sample": f"{n_rows} evenly spaced arrival positions of the slice (grouped SwiGLU "
                      f"expert MLP and gate-weighted un-permute)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="l535b_t8192", choices=sorted(SHAPES))
    ap.add_argument("--simt", action="store_true", help="CUDA-core GEMMs instead of tcgen05")
    ap.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    ap.add_argument("--cpu-tokens", type=int, default=1024)
    ap.add_argument("--ref-tokens", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--expert-backward", action="store_true",
                    help="time the routed experts' backward (moe_expert_ffn_backward) instead")
    ap.add_argument("--backward", action="store_true",
                    help="time the whole layer's backward (moe_backward) instead")
    ap.add_argument("--graph", action="store_true",
                    help="replay one captured CUDA graph of moe_forward per timed step")
    ap.add_argument("--slice", action="store_true",
                    help="time the expert-parallel slice workload (grouped expert MLP + un-permute)")
    ap.add_argument("--all", action="store_true",
                    help="one line per workload (every layer size, fp8 experts, the slice), each "
                         "with the oracle timed on the host cores")
    args = ap.parse_args()
    shape = SHAPES[args.workload]
    if args.impl == "reference":
        run_reference(args, shape)
        return
    if args.expert_backward:
        run_expert_backward(args, shape)
        return
    if args.backward:
        run_layer_backward(args, shape)
        return
    if args.slice:
        run_slice(args)
        return

    import sparse_expert_router_gb300 as m
    m.load()
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    if args.all:
        if world > 1:
            raise SystemExit("--all runs on one GPU")
        run_all(args, m, dev)
        return
    line = bench_forward(args, shape, m, world, rank, local, dev)
    if line is not None:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(shape, args.cpu_tokens, line.pop("_inp"))
        line.pop("_inp", None)
        print(json.dumps(line), flush=True)
    else:
        torch.distributed.destroy_process_group()
        return
    if world > 1:
        torch.distributed.destroy_process_group()


def forward_config(shape, args, world):
    """The `config` object of a forward line (the reference arm prints the same one)."""
    return {"workload": f"{shape.name}: T={shape.T} d={shape.d_model} "
                        f"latent={shape.d_latent} E={shape.n_experts} k={shape.top_k} "
                        f"F={shape.d_ff} shared={shape.n_shared}x{shape.d_ff_shared}"
                        + (f" capacity={shape.capacity[0]}/{shape.capacity[1]}"
                           if shape.capacity else "")
                        + (" zipf" if shape.routing == "zipf" else ""),
            "parallelism": "replicas" if world > 1 else "single GPU",
            "gemm_path": "simt" if args.simt else "tcgen05", "pdl": not args.no_pdl,
            "launch": "cuda graph replay" if args.graph else "eager",
            "expert_weights": shape.expert_dtype,
            "l2": "flushed between timed steps (256 MB write); weights "
                  f"({weight_bytes(shape) / 1e9:.1f} GB) exceed L2"}


def bench_forward(args, shape, m, world, rank, local, dev, e2e_on=None):
    """Times args.steps forwards of `shape` (after the warm-up) and returns rank 0's JSON line as
    a dict (None on the other ranks); "_inp" holds the workload's inputs for the CPU baseline."""
    flags = (m.MOE_FLAG_SIMT if args.simt else 0) | (0 if args.no_pdl else m.MOE_FLAG_PDL)
    cfg = m.LayerConfig.from_shape(shape, flags=flags)
    inp = make_layer_inputs(shape.with_(seed=shape.seed), dev)
    if rank > 0:   # each replica processes its own batch
        inp["x"] = make_layer_inputs(shape.with_(seed=shape.seed + rank, T=shape.T), dev)["x"]
    ws = m.alloc_workspace(cfg, dev)
    y = torch.empty((shape.T, shape.d_model), dtype=shape.torch_dtype, device=dev)
    counts = torch.zeros(shape.n_experts, dtype=torch.int32, device=dev)
    offsets = torch.zeros(shape.n_experts + 1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)     # > L2 (129 MB)
    stream = torch.cuda.current_stream(dev)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(STAGES) + 1)]
    for e in evs:
        e.record(stream)          # creates the CUDA events before their handles are passed on
    aux = {"stage_events": evs, "expert_counts": counts, "expert_offsets": offsets}

    for _ in range(max(3, args.warmup)):
        m.moe_forward(cfg, inp, inp["x"], y, ws, stream=stream, aux=aux)
    torch.cuda.synchronize(dev)
    graph = None
    if args.graph:
        # the whole forward (its kernels, PDL edges and stage events) as one CUDA graph
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            m.moe_forward(cfg, inp, inp["x"], y, ws, stream=torch.cuda.current_stream(dev),
                          aux=aux)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize(dev)
    rep = m.moe_get_device_status(ws)
    if rep["status"] != 0:
        raise RuntimeError(f"device report after warm-up: {rep}")

    clocks = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    step_ms, stage_ms = [], {s: 0.0 for s in STAGES}
    t_wall = time.perf_counter()
    for _ in range(args.steps):
        flush.zero_()                                   # L2 flushed between timed steps
        if graph is not None:
            graph.replay()
        else:
            m.moe_forward(cfg, inp, inp["x"], y, ws, stream=stream, aux=aux)
        evs[-1].synchronize()
        step_ms.append(evs[0].elapsed_time(evs[-1]))
        for i, s in enumerate(STAGES):
            stage_ms[s] += evs[i].elapsed_time(evs[i + 1])
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(sum(step_ms), dev)
    ms_step = total_ms / args.steps
    value = world * shape.T * args.steps / (total_ms / 1e3)

    rep = m.moe_get_device_status(ws)
    if rep["status"] != 0:
        raise RuntimeError(f"device report after the timed steps: {rep}")

    # end to end through the C ABI with host buffers: H2D of x, forward, D2H of y
    e2e = None
    if (not args.no_e2e) if e2e_on is None else e2e_on:
        # the serving path: moe_forward_pipelined over host batches, each batch's input copied in
        # and output copied out inside the timed region, overlapped with the other batches'
        # forwards on two copy streams
        x_host = inp["x"].cpu().pin_memory()
        y_hosts = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
        x_stage = torch.empty((2,) + tuple(inp["x"].shape), dtype=inp["x"].dtype, device=dev)
        y_stage = torch.empty((2,) + tuple(y.shape), dtype=y.dtype, device=dev)
        h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ys = [y_hosts[i % 2] for i in range(args.steps)]
        m.moe_forward_pipelined(cfg, inp, [x_host] * 2, y_hosts, x_stage, y_stage, ws, stream,
                                h2d, d2h)
        torch.cuda.synchronize(dev)
        flush.zero_()
        a.record(stream)
        m.moe_forward_pipelined(cfg, inp, [x_host] * args.steps, ys, x_stage, y_stage, ws,
                                stream, h2d, d2h)
        b.record(stream)
        b.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b), dev)
        y_host = y_hosts[0]
        e2e = {"value": world * shape.T * args.steps / (e2e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
               "d2h_bytes_per_step": y_host.numel() * y_host.element_size()}

    if rank != 0:
        return None

    pk = peaks()
    alg = algorithmic(shape, (offsets[1:] - offsets[:-1]).cpu().tolist())
    # a combine run inside the back GEMM's launch leaves its own stage empty: its bytes are then
    # reported with the back GEMM's stage
    fused = stage_ms["combine"] / args.steps < 0.003 and shape.n_shared > 0
    if fused:
        alg["back_gemm"]["bytes"] += alg.pop("combine")["bytes"]
    stages = {}
    # GEMMs on CUDA cores (the fp32 layer, or --simt) are rated against the fp32 ALU peak
    cuda_core = shape.dtype == "f32" or args.simt
    alu_peak = f32_alu_peak(dev, clk) if cuda_core else None
    for s in STAGES:
        ms = stage_ms[s] / args.steps
        st = {"ms": round(ms, 4)}
        if s == "combine" and fused:
            st["fused_into"] = "back_gemm"
        if s in alg:
            f, by = alg[s]["flops"], alg[s]["bytes"]
            st["gb_s"] = round(by / (ms * 1e-3) / 1e9, 1)
            st["hbm_frac"] = round(st["gb_s"] / pk["hbm_gbs"], 3)
            tr = profiled_traffic(shape.name, s)
            if tr is not None:
                st["traffic"] = tr
            if f and cuda_core:
                st["tflop_s"] = round(f / (ms * 1e-3) / 1e12, 2)
                st["f32_alu_frac"] = round(st["tflop_s"] / alu_peak, 4)
            elif f:
                tp, tps = tc_peak(pk, alg[s]), tc_peak(pk, alg[s], "bf16_sustained")
                st["tflop_s"] = round(f / (ms * 1e-3) / 1e12, 1)
                st[alg[s].get("tc_peak", "bf16") + "_frac"] = round(st["tflop_s"] / tp, 3)
                st[alg[s].get("tc_peak", "bf16") + "_sustained_frac"] = round(st["tflop_s"] / tps, 3)
        stages[s] = st
    dom = max((s for s in STAGES if s in alg), key=lambda s: stage_ms[s])
    f, by = alg[dom]["flops"], alg[dom]["bytes"]
    ms_dom = stage_ms[dom] / args.steps
    tp = alu_peak if cuda_core else tc_peak(pk, alg[dom])
    t_hbm, t_tc = by / (pk["hbm_gbs"] * 1e9), f / (tp * 1e12)
    if cuda_core and t_hbm < t_tc:
        ach = f / (ms_dom * 1e-3) / 1e12
        roof = {"bound": "alu", "achieved": round(ach, 2), "peak": round(tp, 1), "unit": "TFLOP/s",
                "frac": round(ach / tp, 4)}
    elif t_hbm >= t_tc:
        ach = by / (ms_dom * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / pk["hbm_gbs"], 4)}
    else:
        ach = f / (ms_dom * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": round(tp, 1),
                "unit": "TFLOP/s", "frac": round(ach / tp, 4),
                "sustained_frac": round(ach / tc_peak(pk, alg[dom], "bf16_sustained"), 4)}
    roof.update({"kernel": dom, "traffic": profiled_traffic(shape.name, dom),
                 "peak_source": ("derived: SMs x 128 fp32 lanes x 2 flops x max SM clock"
                                 if roof["bound"] == "alu" else pk["source"]
                 + ((" (bf16 burst" + (" x 2, the nominal E4M3/bf16 ratio)"
                                       if alg[dom].get("tc_peak") == "fp8" else ")"))
                    if roof["bound"] == "tensor" else " (HBM copy)"))})
    return {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("f32" if shape.dtype == "f32" else
                  "bf16" if shape.expert_dtype == "bf16" else "bf16; expert MLP e4m3 (f32 accumulate)"),
        "data": "synthetic (seeded N(0,1) activations, N(0,1/fan_in) weights, near-uniform "
                "routing unless the workload is Zipf-skewed)",
        "config": forward_config(shape, args, world),
        "layer_tflop_s": round(sum(shape.flops().values()) / (ms_step * 1e-3) / 1e12, 1),
        "stages": stages,
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": launches_per_forward(shape, args.simt) * args.steps,
        "clocks": clk,
        "wall_s": round(wall, 3),
        "device_report": rep,
        "_inp": inp,
    }


# Every workload of the layer, one JSON line each in --all mode, with the number of tokens of
# the oracle's bounded CPU sample (all threads) and, for the two smallest layers, of a second
# sample timed on one thread.
ALL_WORKLOADS = [("tiny_f32", 256, 256), ("small_bf16", 1024, 128), ("l535b_t8192", 1024, 0),
                 ("l535b_t8192_fp8", 1024, 0), ("l535b_zipf_t16384", 2048, 0),
                 ("l535b_zipf_t16384_cf110", 2048, 0), ("l535b_t65536", 1024, 0)]


def run_all(args, m, dev):
    """One line per workload (the layer at every size, the fp8 expert MLP, the expert-parallel
    slice), each with the oracle timed on the host cores beside it."""
    for name, n_cpu, n_single in ALL_WORKLOADS:
        shape = SHAPES[name]
        line = bench_forward(args, shape, m, 1, 0, 0, dev, e2e_on=False)
        inp = line.pop("_inp")
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(shape, min(n_cpu, shape.T), inp)
            if n_single:
                nt = torch.get_num_threads()
                torch.set_num_threads(1)
                try:
                    line["cpu_baseline_single_core"] = cpu_baseline(shape, n_single, inp)
                finally:
                    torch.set_num_threads(nt)
        print(json.dumps(line), flush=True)
        del inp, line
        torch.cuda.empty_cache()
    run_slice(args)


if __name__ == "__main__":
    main()
