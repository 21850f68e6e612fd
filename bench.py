"""Benchmark of the MXFP4 MoE layer on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one call of the whole layer (router + top-k + tile table + gather/encode
+ gate/up/SwiGLU + down/combine) over one batch of seeded synthetic gpt-oss-shaped
input.  Inputs are resident in HBM when the timed region starts; weight copies are
rotated so that every timed call streams its experts from HBM rather than L2.
Prints one JSON line (rank 0).  For N > 1 (torchrun), every rank runs an independent
replica of the layer (there is no exchange on this path), timings are max-reduced
and `value` is the whole-job throughput.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MXFP4 MoE layer µs/call & tokens/s (batch 1/64/4096), % of HBM roofline"
L2_BYTES = 129 * 1024 * 1024
GATEUP_BYTES_PER_EXPERT = lambda H, I: 2 * I * H // 2 + 2 * I * H // 32   # codes + E8M0 scales
DOWN_BYTES_PER_EXPERT = lambda H, I: H * I // 2 + H * I // 32
GATEUP_FLOPS_PER_ROW = lambda H, I: 2 * 2 * I * H        # one (token, expert) assignment
DOWN_FLOPS_PER_ROW = lambda H, I: 2 * H * I
ACT_TERMS = 4                                            # E2M1 terms of the activation encoding
MXFP4_OVER_BF16 = 13.5 / 2.25                            # nominal dense tensor-rate ratio
DEFAULT_WORKLOAD = "gptoss20b_b1"
NOMINAL_HBM_GBS = 7900.0                                 # GB300 HBM3e, nominal (context beside the measured peak)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="default workload only: skip the batch-64, 120b and prefill lines of the `workloads` block")
    ap.add_argument("--norm", action="store_true",
                    help="RMSNorm + residual fused in front of the layer (moe_forward_norm)")
    ap.add_argument("--eager", action="store_true", help="time eager launches instead of CUDA-graph replays")
    ap.add_argument("--profile", action="store_true",
                    help="minimal run for ncu: no pre-warm, no graphs, no CPU baseline, no clock sampling")
    return ap.parse_args()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smmax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smmax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smmax) if smmax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- traffic from the committed ncu summary
GEMM_HOST_MARKER = b"// ------------------------------------------------------------------ host launchers"


def _code_only(src: bytes) -> bytes:
    """C++ source with comments removed and whitespace collapsed (string literals in
    these files hold no comment markers)."""
    src = re.sub(rb"/\*.*?\*/", b" ", src, flags=re.S)
    src = re.sub(rb"//[^\n]*", b" ", src)
    return re.sub(rb"\s+", b" ", src).strip()


def kernel_source_hash():
    """Hash of the expert GEMM's device code: moe_gemm.cu up to its host launchers,
    and the two headers it draws on, comments and whitespace ignored.  A committed ncu
    summary is used only while this matches the hash recorded with it."""
    import hashlib
    h = hashlib.sha256()
    for fn in ("moe_gemm.cu", "moe_common.cuh", "sm100_ptx.cuh"):
        with open(os.path.join(ROOT, "mxfp4_expert_layer_gb300", "csrc", fn), "rb") as f:
            data = f.read()
        if fn == "moe_gemm.cu" and GEMM_HOST_MARKER in data:
            data = data[:data.index(GEMM_HOST_MARKER)]
        h.update(_code_only(data))
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from profiles/<kernel>_<workload>.md, or None
    when absent or when the kernel source changed since the capture."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    hm = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", txt)
    if not m or not hm or hm.group(1) != kernel_source_hash():
        return None
    return float(m.group(1))


# ---------------------------------------------------------------- CPU oracle baseline
def cpu_baseline(inp, budget_s=12.0, dense=False, max_tokens=8):
    """The oracle as it stands, on the host cores, on a bounded sample of the workload
    (whole passes of the first min(T, max_tokens) tokens until the budget is spent)."""
    import numpy as np
    import oracle
    T = inp.T
    n_tok = min(T, max_tokens)
    tokens = np.arange(n_tok)
    layer = oracle.moe_layer_dense if dense else oracle.moe_layer
    done, t0 = 0, time.perf_counter()
    while True:
        layer(inp, tokens=tokens)
        done += n_tok
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    what = "bf16 experts" if dense else "MXFP4 decode of the touched experts"
    return {"value": done / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{done} tokens of {inp.name} ({n_tok} per pass, full layer incl. {what}) in {dt:.1f} s; "
                      f"numpy, BLAS threads up to {os.cpu_count()}"}


# ---------------------------------------------------------------- distributed plumbing
def dist_init(n):
    """One process per GPU (torchrun env). NCCL on GPUs; gloo where there is no GPU
    (the CPU tests of this plumbing). Replicas exchange only timings."""
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    if world > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(tokens_per_rank, ms_max, world):
    """Whole-job throughput of `world` replicas: every rank's tokens over the slowest
    rank's time per step."""
    return world * tokens_per_rank / (ms_max * 1e-3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- reference arm (the oracle)
def run_reference(args):
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    if rank != 0:
        return
    from synthetic import make_config
    inp = make_config(args.workload)
    import numpy as np
    import oracle
    n_tok = min(inp.T, 8)
    tokens = np.arange(n_tok)
    for _ in range(max(0, min(args.warmup, 1))):
        oracle.moe_layer(inp, tokens=tokens)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.moe_layer(inp, tokens=tokens)
    dt = time.perf_counter() - t0
    val = args.steps * n_tok / dt
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": inp.name, "T": inp.T, "H": inp.H, "I": inp.I, "E": inp.E, "k": inp.k,
                       "sample_tokens_per_step": n_tok},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "kind": "oracle", "cores": os.cpu_count(),
                             "sample": f"{n_tok} tokens of {inp.name} per step, full layer"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ---------------------------------------------------------------- our arm
def bf16_peak_tflops(sustained: bool):
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained" if sustained else "bf16_tflops"]), "measured"
    return (1700.0 if sustained else 1900.0), "fallback"


def main_dense(args):
    """bf16-weight workloads (moe_forward_bf16): Mixtral-8x7B expert shapes."""
    rank, world = dist_init(args.gpus)
    import numpy as np
    import torch

    import mxfp4_expert_layer_gb300 as pkg
    from mxfp4_expert_layer_gb300 import _lib as L
    from synthetic import make_dense_config

    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkg.build()
    L.load()
    inp = make_dense_config(args.workload, seed=rank)
    T, H, I, E, k = inp.T, inp.H, inp.I, inp.E, inp.k
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    x, wr = bf(inp.x), bf(inp.w_router)
    layer = pkg.MoELayerBF16(wr, bf(inp.w_gateup), bf(inp.w_down), k=k)
    if args.no_cpu_baseline:
        del inp.w_gateup, inp.w_down  # host copies are needed only by the CPU baseline
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    layer(x, out=out, topk_idx=idx)
    torch.cuda.synchronize()
    touched = int(torch.unique(idx).numel())
    alg_bytes = touched * 3 * H * I * 2
    flops = 2 * T * k * 3 * H * I
    # weights of one expert set exceed 4x L2 at these shapes: one copy streams from HBM
    copies = max(1, min(8, math.ceil(4 * L2_BYTES / max(alg_bytes, 1))))
    wsets = [(layer.w_gateup, layer.w_down, x)] + [
        (layer.w_gateup.clone(), layer.w_down.clone(), x.clone()) for _ in range(copies - 1)]
    ws = layer.workspace(T)

    def call(i):
        wgu, wd, x_i = wsets[i % copies]
        st = L.moe_forward_bf16(x_i.data_ptr(), wr.data_ptr(), None, wgu.data_ptr(), wd.data_ptr(), T, H, I, E, k,
                                ws.data_ptr(), ws.numel(), out.data_ptr(), None, None,
                                torch.cuda.current_stream().cuda_stream)
        if st != 0:
            raise RuntimeError(f"moe_forward_bf16 failed: {L.moe_error_string(st).decode()}")

    if args.profile:
        for s_ in range(args.warmup + args.steps):
            call(s_)
        torch.cuda.synchronize()
        print(json.dumps({"profile_run": args.workload, "calls": args.warmup + args.steps,
                          "status": layer.device_status(T)}))
        return
    step_calls = copies * math.ceil(4 / copies)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    hx = torch.empty(T, H, dtype=torch.bfloat16, pin_memory=True)
    hx.copy_(x.cpu())
    hout = torch.empty(T, H, dtype=torch.bfloat16, pin_memory=True)
    with torch.cuda.stream(side):
        call(0)
        torch.cuda.synchronize()
        step_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(step_graph, stream=side):
            for j in range(step_calls):
                call(j)
        e2e_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(e2e_graph, stream=side):
            wsets[0][2].copy_(hx, non_blocking=True)
            call(0)
            hout.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    reps = max(1, math.ceil(args.steps / step_calls))
    clocks = ClockSampler(local)
    for _ in range(max(1, math.ceil(args.warmup / step_calls))):
        step_graph.replay()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(reps):
        step_graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(ev0.elapsed_time(ev1) / (reps * step_calls), world)
    clk = clocks.stop()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(args.steps):
        e2e_graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world)
    status = layer.device_status(T)
    if rank != 0:
        return
    hbm, hbm_kind = measured_peaks()
    tc, tc_kind = bf16_peak_tflops(sustained=ms * reps * step_calls > 1000)
    t_hbm, t_tc = alg_bytes / (hbm * 1e9), flops / (tc * 1e12)
    if t_tc > t_hbm:
        ach = flops / (ms * 1e-3) / 1e12
        roof = {"kernel": "whole layer", "bound": "tensor", "achieved": ach, "peak": tc, "unit": "TFLOP/s",
                "frac": ach / tc, "peak_source": f"{tc_kind} bf16", "algorithmic_flops_per_call": flops,
                "traffic": None}
    else:
        ach = alg_bytes / (ms * 1e-3) / 1e9
        roof = {"kernel": "whole layer", "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm, "peak_source": hbm_kind, "algorithmic_bytes_per_call": alg_bytes,
                "traffic": None}
    line = {
        "metric": "bf16-weight MoE layer (Mixtral-8x7B experts) tokens/s", "value": whole_job_tokens_per_s(T, ms, world),
        "unit": "tokens/s", "n_gpus": world, "steps": reps * step_calls, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "T": T, "H": H, "I": I, "E": E, "k": k,
                   "tile_rows": L.moe_tile_rows(T, k, E), "touched_experts": touched,
                   "l2": f"{copies} weight copies, {alg_bytes / 1e9:.2f} GB of experts per call (> 4x L2)",
                   "parallelism": f"replicas x{world}"},
        "us_per_call": ms * 1e3,
        "timing": f"CUDA graphs of {step_calls} consecutive layer calls, replayed",
        "roofline": roof,
        "e2e": {"value": whole_job_tokens_per_s(T, e2e_ms, world), "unit": "tokens/s", "h2d_bytes_per_step": T * H * 2,
                "d2h_bytes_per_step": T * H * 2, "ms_per_step": e2e_ms},
        "gpu_launches": 5 * reps * step_calls,
        "clocks": clk,
        "device_status": status,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, dense=True, max_tokens=2)
    print(json.dumps(line))


STAGE_NAMES = ["route_topk_table", "encode_x", "gateup_swiglu", "down", "combine"]  # MOE_FORWARD_STAGES launches
SIDE_WORKLOADS = ["gptoss20b_b64", "gptoss120b_b64", "gptoss120b_prefill4096"]


def tensor_peaks(L, stream):
    """The measured kind::mxf4 and kind::f16 MMA rates of this GPU (moe_tensor_peak),
    and the rule's MXFP4 figure: the measured bf16 GEMM burst rate times the nominal
    MXFP4/bf16 ratio."""
    import ctypes
    out = {}
    for kind, name in ((L.MOE_PEAK_MXF4, "mxf4_mma_tflops"), (L.MOE_PEAK_BF16, "bf16_mma_tflops")):
        v = ctypes.c_double(0.0)
        st = L.moe_tensor_peak(kind, 20000, ctypes.byref(v), stream)
        out[name] = v.value if st == 0 else None
    bf16, kind = bf16_peak_tflops(sustained=False)
    out["bf16_gemm_tflops"] = bf16
    out["mxf4_rule_tflops"] = bf16 * MXFP4_OVER_BF16
    out["rule_source"] = f"{kind} cuBLAS bf16 burst x nominal mxfp4/bf16 ratio ({MXFP4_OVER_BF16:g})"
    return out


def stage_bytes_and_flops(T, H, I, E, k, touched):
    """Algorithmic bytes (and FLOPs) of each launch of one layer call."""
    b = {"route_topk_table": E * H * 2 + T * H * 2,
         "encode_x": T * H * 2 + T * k * H * (ACT_TERMS // 2 + 1 / 8),
         "gateup_swiglu": touched * GATEUP_BYTES_PER_EXPERT(H, I),
         "down": touched * DOWN_BYTES_PER_EXPERT(H, I),
         "combine": T * k * H * 4 + T * H * 2}
    f = {"gateup_swiglu": GATEUP_FLOPS_PER_ROW(H, I) * T * k, "down": DOWN_FLOPS_PER_ROW(H, I) * T * k}
    return b, f


def measure_layer(args, wl, rank, world, dev, stream_peaks, headline, steps):
    """Everything measured for one MXFP4 workload: the graph-timed layer, eager
    launches, the per-launch split, the roofline of the dominant launch, the tensor
    pipe of the expert GEMMs and (headline only) the end-to-end number."""
    import numpy as np
    import torch

    import mxfp4_expert_layer_gb300 as pkg
    from mxfp4_expert_layer_gb300 import _lib as L
    from synthetic import make_config

    inp = make_config(wl, seed=rank)
    T, H, I, E, k = inp.T, inp.H, inp.I, inp.E, inp.k
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    x = to(inp.x.view(np.int16)).view(torch.bfloat16)
    wr = to(inp.w_router.view(np.int16)).view(torch.bfloat16)
    bias = None if inp.router_bias is None else to(inp.router_bias)
    layer = pkg.MoELayer.from_mxfp4(wr, to(inp.gu_codes), to(inp.gu_scales), to(inp.dn_codes), to(inp.dn_scales),
                                    k=k, router_bias=bias)
    if not headline or args.no_cpu_baseline:
        del inp.gu_codes, inp.gu_scales, inp.dn_codes, inp.dn_scales  # only the CPU baseline reads them
    # routing of the workload (same for every call): touched experts give the algorithmic bytes
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    wts = torch.empty(T, k, dtype=torch.float32, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    layer(x, out=out, topk_idx=idx, topk_w=wts)
    torch.cuda.synchronize()
    touched = int(torch.unique(idx).numel())
    sbytes, sflops = stage_bytes_and_flops(T, H, I, E, k, touched)
    alg_bytes = sbytes["gateup_swiglu"] + sbytes["down"]

    # rotate copies of the whole layer input (expert weights, router weight, x) so the
    # touched experts of every call come from HBM and nothing a real model would not
    # find in L2 (another layer's router, another step's activations) is found there
    copies = max(1, min(16, math.ceil(4 * L2_BYTES / max(alg_bytes, 1))))
    norm = args.norm and headline
    if norm:
        from synthetic import make_norm_inputs
        r_np, g_np, eps = make_norm_inputs(T, H, seed=rank)
        resid = to(r_np.view(np.int16)).view(torch.bfloat16)
        gamma = to(g_np.view(np.int16)).view(torch.bfloat16)
        res_out = torch.empty_like(x)
    else:
        resid = x  # unused
    wsets = [(layer.w_gateup, layer.w_down, wr, x, resid)] + [
        (layer.w_gateup.clone(), layer.w_down.clone(), wr.clone(), x.clone(), resid.clone())
        for _ in range(copies - 1)]
    ws = layer.workspace(T)

    def call(i, events=None, with_norm=norm):
        wgu, wd, wr_i, x_i, r_i = wsets[i % copies]
        b = None if bias is None else bias.data_ptr()
        cs = torch.cuda.current_stream().cuda_stream
        if with_norm and events is None:
            st = L.moe_forward_norm(x_i.data_ptr(), r_i.data_ptr(), gamma.data_ptr(), eps, wr_i.data_ptr(), b,
                                    wgu.data_ptr(), wd.data_ptr(), T, H, I, E, k, 0, ws.data_ptr(), ws.numel(),
                                    out.data_ptr(), res_out.data_ptr(), None, None, cs)
        elif events is None:
            st = L.moe_forward(x_i.data_ptr(), wr_i.data_ptr(), b, wgu.data_ptr(), wd.data_ptr(), T, H, I, E, k,
                               ws.data_ptr(), ws.numel(), out.data_ptr(), None, None, cs)
        else:
            st = L.moe_forward_timed(x_i.data_ptr(), wr_i.data_ptr(), b, wgu.data_ptr(), wd.data_ptr(), T, H, I, E,
                                     k, ws.data_ptr(), ws.numel(), out.data_ptr(), None, None, events, cs)
        if st != 0:
            raise RuntimeError(f"moe_forward failed: {L.moe_error_string(st).decode()}")

    launches = L.moe_forward_launches(T, H, I, E, k)
    if args.profile:
        for s_ in range(args.warmup + steps):
            call(s_)
        torch.cuda.synchronize()
        return {"profile_run": inp.name, "calls": args.warmup + steps, "status": layer.device_status(T)}

    # the layer runs inside a captured decode step in the pages' engine: one CUDA
    # graph holds the calls of every weight copy in sequence (consecutive layers of
    # a step, each with its own weights), so a layer's first launch overlaps the
    # previous layer's last as it would in that step.  Single-call graphs serve the
    # remainder of K steps and the per-launch split; --eager times plain launches.
    nk = len(STAGE_NAMES)
    step_calls = copies * math.ceil(8 / copies)  # layer calls per step graph: >= 8, whole rotations
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graphs, tgraphs, tevents, e2e_graphs = [], [], [], []
    if headline:
        hx = torch.empty(T, H, dtype=torch.bfloat16, pin_memory=True)
        hx.copy_(x.cpu())
        hr = torch.empty(T, H, dtype=torch.bfloat16, pin_memory=True)
        hr.copy_(resid.cpu())
        hout = torch.empty(T, H, dtype=torch.bfloat16, pin_memory=True)
    with torch.cuda.stream(side):
        call(0)
        torch.cuda.synchronize()
        for j in range(copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                call(j)
            graphs.append(g)
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
            for e in evs:
                e.record(side)
            torch.cuda.synchronize()
            tg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(tg, stream=side):
                call(j, ctypes_array(evs))
            tgraphs.append(tg)
            tevents.append(evs)
            if headline:
                eg = torch.cuda.CUDAGraph()
                with torch.cuda.graph(eg, stream=side):
                    wsets[j][3].copy_(hx, non_blocking=True)
                    if norm:
                        wsets[j][4].copy_(hr, non_blocking=True)
                    call(j)
                    hout.copy_(out, non_blocking=True)
                e2e_graphs.append(eg)
        step_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(step_graph, stream=side):
            for j in range(step_calls):
                call(j)
        if norm:
            # the same step without the norm step, for its cost
            plain_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(plain_graph, stream=side):
                for j in range(step_calls):
                    call(j, with_norm=False)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step(i):
        if args.eager:
            call(i)
        else:
            graphs[i % copies].replay()

    def run_steps(n):
        # n layer calls: whole multi-call graphs, then single-call graphs for the rest
        if args.eager:
            for s_ in range(n):
                call(s_)
            return
        for _ in range(n // step_calls):
            step_graph.replay()
        for s_ in range(n % step_calls):
            graphs[s_ % copies].replay()

    # pre-warm: bring clocks up (~0.5 s of steps), then the W warm-up steps
    t_end = time.perf_counter() + 0.5
    i = 0
    while time.perf_counter() < t_end:
        for _ in range(20):
            step(i)
            i += 1
        torch.cuda.synchronize()
    run_steps(args.warmup)
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    run_steps(steps)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = ev0.elapsed_time(ev1) / steps
    ms = max_over_ranks(ms, world)
    i += steps

    res = {"inp": inp, "T": T, "H": H, "I": I, "E": E, "k": k, "touched": touched, "copies": copies,
           "step_calls": step_calls, "alg_bytes": alg_bytes, "ms": ms, "launches": launches}
    if norm:
        torch.cuda.synchronize()
        reps_p = max(1, steps // step_calls)
        ev0.record(stream)
        for _ in range(reps_p):
            plain_graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        res["plain_us"] = ev0.elapsed_time(ev1) * 1e3 / (reps_p * step_calls)

    # eager launches, for reference (host launch overhead included)
    torch.cuda.synchronize()
    ev0.record(stream)
    for s_ in range(steps):
        call(i + s_)
    ev1.record(stream)
    torch.cuda.synchronize()
    res["eager_ms"] = ev0.elapsed_time(ev1) / steps

    # per-launch split: single-call graphs with an event between consecutive launches
    # (the event breaks the programmatic-launch overlap, so each launch is timed alone)
    per_kernel = [0.0] * nk
    reps = max(1, steps // copies)
    for r in range(reps):
        for j in range(copies):
            tgraphs[j].replay()
            torch.cuda.synchronize()
            for q in range(nk):
                per_kernel[q] += tevents[j][q].elapsed_time(tevents[j][q + 1])
    per_kernel = {n: v / (reps * copies) for n, v in zip(STAGE_NAMES, per_kernel)}
    res["per_kernel_ms"] = per_kernel

    hbm, hbm_kind = measured_peaks()
    mx = stream_peaks["mxf4_mma_tflops"] or stream_peaks["mxf4_rule_tflops"]
    mx_src = "measured kind::mxf4 MMA rate (moe_tensor_peak)" if stream_peaks["mxf4_mma_tflops"] else \
        stream_peaks["rule_source"]
    # the dominant launch (longest single-launch time) and the roof that binds it: its
    # algorithmic bytes at the HBM peak, or (expert GEMMs) the MMAs it issues
    # (ACT_TERMS per product) at the measured MXFP4 rate
    dom = max(per_kernel, key=per_kernel.get)
    dom_ms = per_kernel[dom]
    t_hbm = sbytes[dom] / (hbm * 1e9)
    t_tc = sflops.get(dom, 0) * ACT_TERMS / (mx * 1e12)
    if t_tc > t_hbm:
        achieved = sflops[dom] / (dom_ms * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": mx, "unit": "TFLOP/s",
                "frac": achieved / mx, "peak_source": mx_src,
                "frac_of_bf16_x6": achieved / stream_peaks["mxf4_rule_tflops"],
                "issued_frac": achieved * ACT_TERMS / mx,
                "algorithmic_flops_per_launch": sflops[dom], "launch_us": dom_ms * 1e3,
                "traffic": committed_traffic(dom, inp.name)}
    else:
        achieved = sbytes[dom] / (dom_ms * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "peak_source": hbm_kind,
                "algorithmic_bytes_per_launch": sbytes[dom], "launch_us": dom_ms * 1e3,
                "traffic": committed_traffic(dom, inp.name)}
    res["roofline"] = roof
    gemm_ms = per_kernel["gateup_swiglu"] + per_kernel["down"]
    fl = sum(sflops.values())
    res["tensor_pipe"] = {"algorithmic_tflops": fl / (gemm_ms * 1e-3) / 1e12,
                          "issued_tflops": ACT_TERMS * fl / (gemm_ms * 1e-3) / 1e12,
                          "mxf4_peak_tflops": mx, "peak_source": mx_src,
                          "algorithmic_frac": fl / (gemm_ms * 1e-3) / 1e12 / mx,
                          "issued_frac": ACT_TERMS * fl / (gemm_ms * 1e-3) / 1e12 / mx,
                          "algorithmic_frac_of_bf16_x6": fl / (gemm_ms * 1e-3) / 1e12 / stream_peaks["mxf4_rule_tflops"],
                          "note": f"expert GEMMs (gate/up + down launches); each product is issued as {ACT_TERMS} "
                                  f"E2M1-term MMAs"}

    if headline:
        # end to end through the C ABI: pinned host input -> device, layer, device -> pinned host
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s_ in range(steps):
            e2e_graphs[(i + s_) % copies].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        res["e2e_ms"] = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    res["status"] = layer.device_status(T)
    return res


def main():
    args = parse()
    if args.workload.startswith("mixtral") or args.workload.startswith("dense"):
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the bf16-weight workloads have no reference "
                              "arm; their parity is checked against the oracle in tests/test_gpu_dense.py"}))
            return
        return main_dense(args)
    if args.impl == "reference":
        return run_reference(args)
    rank, world = dist_init(args.gpus)
    import torch

    import mxfp4_expert_layer_gb300 as pkg
    from mxfp4_expert_layer_gb300 import _lib as L

    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkg.build()
    L.load()
    peaks = tensor_peaks(L, torch.cuda.current_stream().cuda_stream)
    if args.profile:
        print(json.dumps(measure_layer(args, args.workload, rank, world, dev, peaks, True, args.steps)))
        return
    clocks = ClockSampler(local)
    r = measure_layer(args, args.workload, rank, world, dev, peaks, True, args.steps)
    side = {}
    if args.workload == DEFAULT_WORKLOAD and not args.no_workloads:
        for wl in SIDE_WORKLOADS:
            torch.cuda.empty_cache()
            w = measure_layer(args, wl, rank, world, dev, peaks, False, min(args.steps, 100))
            side[wl] = {"us_per_call": w["ms"] * 1e3,
                        "tokens_per_s": whole_job_tokens_per_s(w["T"], w["ms"], world),
                        "touched_experts": w["touched"],
                        "layer_hbm_gbs": w["alg_bytes"] / (w["ms"] * 1e-3) / 1e9,
                        "layer_roofline_frac": w["alg_bytes"] / (w["ms"] * 1e-3) / 1e9 / measured_peaks()[0],
                        "per_kernel_us": {n: v * 1e3 for n, v in w["per_kernel_ms"].items()},
                        "roofline": w["roofline"], "tensor_pipe": w["tensor_pipe"], "device_status": w["status"],
                        "timing": f"CUDA graphs of {w['step_calls']} consecutive layer calls cycling over "
                                  f"{w['copies']} weight copies, replayed; {min(args.steps, 100)} calls"}
            del w
    clk = clocks.stop()
    if rank != 0:
        return
    inp, T, H, I, E, k = r["inp"], r["T"], r["H"], r["I"], r["E"], r["k"]
    ms, alg_bytes, copies, step_calls = r["ms"], r["alg_bytes"], r["copies"], r["step_calls"]
    peak, peak_kind = measured_peaks()
    us = ms * 1e3
    line = {
        "metric": METRIC, "value": whole_job_tokens_per_s(T, ms, world), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "mxfp4",
        "dtype_detail": "tcgen05 kind::mxf4: E2M1 weights x E2M1 activations (4 terms), E8M0 block scales, "
                        "f32 accumulate, bf16 out",
        "data": "synthetic",
        "config": {"workload": inp.name, "T": T, "H": H, "I": I, "E": E, "k": k,
                   "tile_rows": L.moe_tile_rows(T, k, E), "touched_experts": r["touched"],
                   "l2": f"{copies} rotating copies of weights, router weight and x "
                         f"({copies * alg_bytes / 1e6:.0f} MB of experts touched per rotation > 4x L2)",
                   "parallelism": f"replicas x{world}"},
        "us_per_call": us,
        "timing": "eager launches" if args.eager else
                  f"CUDA graphs of {step_calls} consecutive layer calls cycling over {copies} weight "
                  f"copies, replayed",
        "eager_us_per_call": r["eager_ms"] * 1e3,
        "layer_hbm_gbs": alg_bytes / (ms * 1e-3) / 1e9,
        "layer_roofline_frac": alg_bytes / (ms * 1e-3) / 1e9 / peak,
        "layer_frac_of_nominal_hbm": alg_bytes / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
        "per_kernel_us": {n: v * 1e3 for n, v in r["per_kernel_ms"].items()},
        "per_kernel_note": "each launch timed alone: single-call graphs with an event between consecutive "
                           "launches, which removes the programmatic-launch overlap the layer runs with",
        "roofline": r["roofline"],
        "tensor_pipe": r["tensor_pipe"],
        "tensor_peaks": peaks,
        "e2e": {"value": whole_job_tokens_per_s(T, r["e2e_ms"], world), "unit": "tokens/s",
                "h2d_bytes_per_step": T * H * 2 * (2 if args.norm else 1),
                "d2h_bytes_per_step": T * H * 2, "ms_per_step": r["e2e_ms"]},
        "gpu_launches": r["launches"] * args.steps,
        "clocks": clk,
        "device_status": r["status"],
    }
    if side:
        line["workloads"] = side
    if args.norm:
        line["config"]["norm"] = "RMSNorm + residual fused in front of the layer (moe_forward_norm)"
        line["norm_step"] = {"us_per_call_without_norm": r["plain_us"], "added_us": us - r["plain_us"],
                             "per_kernel_note": "per_kernel_us and roofline come from the layer's timed "
                                                "graphs without the norm step"}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp)
    print(json.dumps(line))


def ctypes_array(events):
    import ctypes
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    return arr


if __name__ == "__main__":
    main()
