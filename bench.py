"""Benchmark of the fused grouped expert MLP (route + forward + backward) on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

One step = one pass of the whole hot path over one batch of synthetic tokens: route + permute,
FC1 + GLU + prob scale, FC2, combine, dY gather, FC2 dgrad + dGLU, FC2 wgrad, FC1 dgrad,
dx combine, FC1 wgrad. The default workload is the Mixtral-8x7B-shaped BF16 layer
(T=8192, E=8, top-2, H=4096, F=14336, SwiGLU). Inputs are resident in HBM before timing;
every step reads ~2.8 GB of weights and writes ~2.8 GB of weight gradients, far above the
129 MB L2, so no explicit flush is needed. Prints one JSON line (rank 0).

Multi-GPU: the layer runs as independent replicas, one per rank (no data-path collective);
`value` is the sum over ranks of the work divided by the slowest rank's time.

--impl reference times the fp64 CPU oracle on a bounded sample of the same workload on the
host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# the CPU baseline (the fp64 oracle) uses every host core: BLAS threads are set explicitly,
# before numpy loads its BLAS
HOST_CORES = os.cpu_count() or 1
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(HOST_CORES))

import numpy as np  # noqa: E402

from grouped_gemm_device_gb300 import synth  # noqa: E402

METRIC = "grouped-MLP fwd+bwd TFLOPS & tokens/s at 1 GB300; % of tensor-core peak"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="mixtral_bf16", choices=sorted(synth.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sm-margin", type=int, default=0)
    ap.add_argument("--tokens", type=int, default=0, help="override T (profiling runs)")
    ap.add_argument("--experts", type=int, default=0, help="override E (profiling runs)")
    ap.add_argument("--overlap-sweep", default="",
                    help="comma-separated SM margins: time the layer step, a concurrent "
                         "memory-bound job (device copies on another stream) and both "
                         "together at each margin; prints one JSON line")
    ap.add_argument("--extras", type=int, default=0,
                    help="epilogue extras bits: 1 FC1 bias, 2 feature scale (BF16 gated)")
    ap.add_argument("--recompute", action="store_true",
                    help="keep no FC1 output; the FC2-dgrad kernel recomputes it")
    ap.add_argument("--workloads", default="auto",
                    help="extra workloads timed after the headline one, each with its own "
                         "entry under 'workloads': 'auto' (every other configuration when the "
                         "headline is the default one), 'none', or a comma-separated list")
    ap.add_argument("--workload-steps", type=int, default=20)
    ap.add_argument("--no-pdl-compare", dest="pdl_compare", action="store_false",
                    help="skip timing the step with and without programmatic dependent launch")
    ap.add_argument("--e2e-pdl", action="store_true",
                    help="run the end-to-end pass with programmatic dependent launch (default: "
                         "ordinary stream order, measured as fast or faster)")
    return ap.parse_args()


def config_of(args):
    cfg = synth.CONFIGS[args.config]
    if args.tokens:
        cfg = cfg.with_(T=args.tokens, name=cfg.name + f"_T{args.tokens}")
    if args.experts:
        cfg = cfg.with_(E=args.experts, k=min(cfg.k, args.experts),
                        name=cfg.name + f"_E{args.experts}")
    return cfg


def workload_name(cfg) -> str:
    return (f"{cfg.name}: T={cfg.T} E={cfg.E} top-{cfg.k} H={cfg.H} F={cfg.F} "
            f"{cfg.activation} {cfg.precision}")


def gemm_flops(cfg, recompute=False):
    """Executed flops per GEMM launch (with recomputation the FC2-dgrad kernel also rebuilds
    the FC1 output); the step metric counts the model's flops only."""
    R = cfg.R
    H, F, N1 = cfg.H, cfg.F, cfg.N1
    return {
        "gemm_fc1_fprop": 2.0 * R * H * N1, "gemm_fc2_fprop": 2.0 * R * F * H,
        "gemm_fc2_dgrad": 2.0 * R * H * F + (2.0 * R * H * N1 if recompute else 0.0),
        "gemm_fc2_wgrad": 2.0 * R * F * H,
        "gemm_fc1_dgrad": 2.0 * R * N1 * H, "gemm_fc1_wgrad": 2.0 * R * H * N1,
    }


# launches of one kernel that recur within a step, named by their order in the step
REPEATED = {
    "mxfp8_quantize": ("mxfp8_quant_x", "mxfp8_quant_w1", "mxfp8_quant_w2", "mxfp8_quant_dy"),
    "nvfp4_quantize": ("nvfp4_quant_x", "nvfp4_quant_w1", "nvfp4_quant_w2", "nvfp4_quant_a",
                       "nvfp4_quant_dy", "nvfp4_quant_dz"),
    "nvfp4_amax": ("nvfp4_amax_w1", "nvfp4_amax_w2"),
}
# dense tensor-core rate of the operand type relative to bf16 (nominal: fp8 4.5 and fp4
# 13.5 PFLOP/s against bf16's 2.25)
TENSOR_RATIO = {"bf16": 1.0, "mxfp8": 2.0, "nvfp4": 6.0}
# GB300 nominal dense tensor peaks (TFLOP/s) and HBM3e bandwidth (GB/s), for context beside
# the measured denominators
NOMINAL_TFLOPS = {"bf16": 2250.0, "mxfp8": 4500.0, "nvfp4": 13500.0}
NOMINAL_HBM_GBS = 7900.0
# weight quantisation kernels of a step (re-run from the BF16 masters by every forward unless
# the forward reuses the copies)
WEIGHT_QUANT = ("mxfp8_quant_w1", "mxfp8_quant_w2", "nvfp4_quant_w1", "nvfp4_quant_w2",
                "nvfp4_amax_w1", "nvfp4_amax_w2")
HEADLINE = "mixtral_bf16"
# the other workloads a default run times too (Mixtral MXFP8, DeepSeek-V3 MXFP8, GPT-OSS BF16
# and MXFP8 with the activation sweep, NVFP4)
EXTRA_WORKLOADS = ("mixtral_mxfp8", "dsv3_mxfp8", "gptoss_bf16", "gptoss_mxfp8",
                   "gptoss_geglu_bf16", "gptoss_srelu_bf16", "gptoss_geglu_mxfp8",
                   "gptoss_srelu_mxfp8", "mixtral_nvfp4", "gptoss_nvfp4")
DTYPE = {"bf16": "bf16", "mxfp8": "e4m3+e8m0 (fp32 accumulate)",
         "nvfp4": "e2m1+e4m3+fp32 scale (fp32 accumulate)"}


def kernel_bytes(cfg, recompute=False):
    """Algorithmic HBM bytes per launch: each operand read once, each result written once
    (R = routed rows; MXFP8 data is 1 byte plus one scale byte per 32, NVFP4 half a byte plus
    one scale byte per 16). With recomputation the FC1 kernel writes no Z and the FC2-dgrad
    kernel reads X and W1 (their quantised copies in MXFP8 and NVFP4) instead of Z."""
    R, T, E = cfg.R, cfg.T, cfg.E
    H, F, N1 = cfg.H, cfg.F, cfg.N1
    R_cap = cfg.R_cap
    common = {
        "gather_x": R_cap * H * 2 + R * H * 2, "gather_dy": R_cap * H * 2 + R * H * 2,
        "combine_y": R * H * 2 + T * H * 2, "combine_dx": R * H * 2 + T * H * 2,
    }
    if cfg.precision == "bf16":
        s = 2.0
        out = {"gemm_fc1_fprop": R * H * s + E * N1 * H * s + R * N1 * 2 + R * F * 2,
               "gemm_fc2_dgrad": R * H * s + E * F * H * s + R * N1 * 2 + R * N1 * 2}
    elif cfg.precision == "nvfp4":
        s = 0.5 + 1.0 / 16.0
        out = {"gemm_fc1_fprop": R * H * s + E * N1 * H * s + R * N1 * 2 + R * F * 2,
               "gemm_fc2_dgrad": R * H * s + E * F * H * s + R * N1 * 2 + R * N1 * 2,
               # bf16 in, row-wise and transposed copies out
               "nvfp4_quant_x": R_cap * H * (2 + 2 * s), "nvfp4_quant_dy": R_cap * H * (2 + 2 * s),
               "nvfp4_quant_a": R_cap * F * (2 + 2 * s),
               "nvfp4_quant_dz": R_cap * N1 * (2 + 2 * s),
               "nvfp4_quant_w1": E * N1 * H * (2 + 2 * s),
               "nvfp4_quant_w2": E * F * H * (2 + 2 * s),
               "nvfp4_amax_w1": E * N1 * H * 2, "nvfp4_amax_w2": E * F * H * 2}
    else:  # mxfp8: the fused epilogues write the quantised A and dZ copies (both directions)
        s = 33.0 / 32.0
        out = {"gemm_fc1_fprop": R * H * s + E * N1 * H * s + R * N1 * 2 + 2 * R * F * s,
               "gemm_fc2_dgrad": R * H * s + E * F * H * s + R * N1 * 2 + 2 * R * N1 * s,
               "mxfp8_quant_x": R_cap * H * (2 + 2 * s), "mxfp8_quant_dy": R_cap * H * (2 + 2 * s),
               "mxfp8_quant_w1": E * N1 * H * (2 + 2 * s),
               "mxfp8_quant_w2": E * F * H * (2 + 2 * s)}
    out.update({
        "gemm_fc2_fprop": R * F * s + E * F * H * s + R * H * 2,
        "gemm_fc2_wgrad": R * F * s + R * H * s + E * F * H * 2,
        "gemm_fc1_dgrad": R * N1 * s + E * N1 * H * s + R * H * 2,
        "gemm_fc1_wgrad": R * N1 * s + R * H * s + E * N1 * H * 2,
    })
    if recompute:  # no Z written or read; X and W1 read a second time
        out["gemm_fc1_fprop"] -= R * N1 * 2
        out["gemm_fc2_dgrad"] += R * H * s + E * N1 * H * s - R * N1 * 2
    out.update(common)
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------------- distributed
def dist_backend() -> str:
    """nccl for GPU replicas; gloo where no GPU is visible (the host-side path is tested that
    way). MOE_DIST_BACKEND overrides."""
    import torch
    return os.environ.get("MOE_DIST_BACKEND") or ("nccl" if torch.cuda.is_available() else "gloo")


def dist_setup(args=None):
    """Join the process group torchrun describes (WORLD_SIZE, RANK, LOCAL_RANK, MASTER_*);
    one process per GPU, each an independent replica of the layer."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        backend = dist_backend()
        if backend == "nccl":
            torch.cuda.set_device(local)
        if not dist.is_initialized():
            dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(v: float, ws: int) -> float:
    """The slowest rank's value: the job's step time is the max over replicas."""
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, ms_max: float, world: int) -> float:
    """Weak scaling: every rank processes the same units; the job's rate is all ranks' units
    over the slowest rank's time."""
    return units_per_rank * world / (ms_max / 1e3)


# ------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if re.match(r"^[\d.]+$", r[1])]
        mx = [float(r[2]) for r in rows if re.match(r"^[\d.]+$", r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------------- inputs
def host_inputs(cfg):
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        w1 = list(ex.map(lambda e: synth.gen_w1_expert(cfg, e), range(cfg.E)))
        w2 = list(ex.map(lambda e: synth.gen_w2_expert(cfg, e), range(cfg.E)))
    return dict(logits=synth.gen_logits(cfg), x=synth.gen_x(cfg), dy=synth.gen_dy(cfg), w1=w1,
                w2=w2)


def traffic_for(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu table for the
    workload, if it was taken on the current kernel source (the table records the sha256 of
    gemm.cu it was measured on); None otherwise."""
    path = os.path.join(ROOT, "profiles", f"gemm_dram_traffic_{workload}.txt")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m_sha = re.search(r"(\w+\.cu) sha256\[:16\]:\s*(\w+)", txt)
    m_b = re.search(rf"^{re.escape(kernel)}\s+[\d.]+\s+[\d.]+\s+(\d+)", txt, re.M)
    if not m_sha or not m_b:
        return None
    src = os.path.join(ROOT, "grouped_gemm_device_gb300", "csrc", m_sha.group(1))
    if not os.path.exists(src):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if m_sha.group(2) != sha:
        return None
    return float(m_b.group(1))


# ------------------------------------------------------------------------- CPU oracle
def oracle_sample(cfg, rows: int, inputs=None):
    """fp64 oracle forward+backward of expert 0 on `rows` of its routed tokens. Returns
    (seconds, flops, description); weights are converted outside the timed part."""
    from oracle import moe as om
    lg = inputs["logits"] if inputs else synth.gen_logits(cfg)
    ids, probs = om.route(lg, cfg.k)
    tok, slot = np.nonzero(ids == 0)
    tok, slot = tok[:rows], slot[:rows]
    xb = inputs["x"] if inputs else synth.gen_x(cfg)
    dyb = inputs["dy"] if inputs else synth.gen_dy(cfg)
    w1b = inputs["w1"][0] if inputs else synth.gen_w1_expert(cfg, 0)
    w2b = inputs["w2"][0] if inputs else synth.gen_w2_expert(cfg, 0)
    X, dY = om.bf16_to_f64(xb[tok]), om.bf16_to_f64(dyb[tok])
    W1, W2 = om.bf16_to_f64(w1b), om.bf16_to_f64(w2b)
    p = probs[tok, slot]
    act = om.ActParams(cfg.activation, cfg.beta, cfg.gate_max, cfg.lin_lo, cfg.lin_hi,
                       cfg.lin_offset)
    mx = cfg.precision == "mxfp8"
    t0 = time.perf_counter()
    if cfg.precision == "nvfp4":
        # the stage-by-stage NVFP4 oracle on a one-expert layer made of these rows (every
        # quantisation of expert 0's operands included)
        om.layer_nvfp4(np.zeros((len(tok), 1), np.float32), X, W1[None], W2[None], 1, act,
                       synth.gen_rht_mask(cfg), dy=dY, align=cfg.align)
        kind = "NVFP4 oracle (one-expert layer)"
    else:
        Z, a, a_s, Y = om.expert_forward(X, W1, W2, p, act, mx)
        om.expert_backward(X, W1, W2, p, Z, a, a_s, dY, act, mx)
        kind = "oracle"
    dt = time.perf_counter() - t0
    n = len(tok)
    flops = 3.0 * (2.0 * n * cfg.H * cfg.N1 + 2.0 * n * cfg.F * cfg.H)
    desc = (f"{kind} fp64 fwd+bwd of expert 0 on {n} routed tokens of {cfg.name} "
            f"({flops / 1e9:.0f} GFLOP)")
    return dt, flops, desc, n


def blas_threads() -> int:
    """BLAS threads in use: threadpoolctl's report where it is installed, else the thread
    count this script set for OpenBLAS before numpy loaded."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return int(os.environ.get("OPENBLAS_NUM_THREADS", HOST_CORES))


def tensor_peak(peaks, precision, clocks):
    """Tensor roofline of the operand type at the clock the timed region held: the measured
    bf16 burst rate x the nominal operand-type ratio x (median SM clock / max SM clock).
    Returns (TFLOP/s, description)."""
    burst = peaks.get("bf16_tflops", 1900.0)
    ratio = TENSOR_RATIO[precision]
    scale = 1.0
    if clocks and clocks.get("sm_mhz") and clocks.get("sm_max_mhz"):
        scale = min(1.0, clocks["sm_mhz"] / clocks["sm_max_mhz"])
    kind = (f"bf16_tflops (burst) x {ratio:g} ({precision}/bf16 nominal ratio) x "
            f"{scale:.3f} (median/max SM clock)")
    return burst * ratio * scale, kind


def run_reference(args):
    ws, rank, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return
    cfg = config_of(args)
    inputs = {"logits": synth.gen_logits(cfg), "x": synth.gen_x(cfg), "dy": synth.gen_dy(cfg),
              "w1": [synth.gen_w1_expert(cfg, 0)], "w2": [synth.gen_w2_expert(cfg, 0)]}
    rows = 128
    for _ in range(args.warmup):
        oracle_sample(cfg, 32, inputs)
    tot_t = tot_f = 0.0
    desc = ""
    tokens = 0
    for _ in range(args.steps):
        dt, fl, desc, n = oracle_sample(cfg, rows, inputs)
        tot_t += dt
        tot_f += fl
        tokens += n
    value = tot_f / tot_t / 1e12
    cores = blas_threads()
    world_n = int(os.environ.get("WORLD_SIZE", "1"))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": max(args.gpus, world_n), "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(cfg), "sample": desc},
        "tokens_per_s": tokens / tot_t,
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "host_cpu_count": HOST_CORES, "blas_threads": cores,
                         "sample": f"per step: {desc}"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------- our arm
def overlap_sweep(args):
    """[NV-blog] 'configurable SM margin': the persistent GEMMs leave `margin` SMs to other
    kernels. For each margin, time K layer steps alone, a memory-bound job alone (repeated
    1 GiB device copies on a second stream), and both started together; 'hidden' is the share
    of the job's own time that the overlap removed."""
    import torch

    import grouped_gemm_device_gb300 as g
    from grouped_gemm_device_gb300 import build as gbuild

    gbuild.build()
    g.load()
    cfg = config_of(args)
    margins = [int(m) for m in args.overlap_sweep.split(",") if m.strip()]
    hin = host_inputs(cfg)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)

    dev = torch.device("cuda", 0)
    w1_log = torch.stack([bf(w) for w in hin["w1"]]).to(dev)
    w1p = g.pack_w1(w1_log, gated=cfg.gated, ilv=cfg.ilv)
    del w1_log
    w2 = torch.stack([bf(w) for w in hin["w2"]]).to(dev)
    logits = torch.from_numpy(hin["logits"]).to(dev)
    x = bf(hin["x"]).to(dev)
    dy = bf(hin["dy"]).to(dev)
    # the concurrent job: a 1 GiB device-to-device copy (short-lived blocks, like the
    # communication kernels the margin is meant for)
    src = torch.empty(1 << 30, dtype=torch.uint8, device=dev).fill_(1)
    dst = torch.empty_like(src)
    side = torch.cuda.Stream()
    main_s = torch.cuda.current_stream()
    steps = max(3, args.steps)

    def timed(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        fn()
        main_s.wait_stream(side)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    out = []
    for m in margins:
        layer = g.MoELayer(g.desc_from_config(cfg, sm_margin=m), dev)

        def layer_steps():
            for _ in range(steps):
                layer.route_permute(logits, x, cfg.T)
                layer.forward(w1p, w2, cfg.T)
                layer.backward(dy, w1p, w2, cfg.T)

        def job(n):
            side.wait_stream(main_s)
            with torch.cuda.stream(side):
                for _ in range(n):
                    dst.copy_(src, non_blocking=True)

        layer_steps()  # warm-up (and the kernels' one-time set-up)
        t_layer = timed(layer_steps)
        t_one = timed(lambda: job(1))
        n_job = max(1, int(round(0.8 * t_layer / max(t_one, 1e-3))))
        t_job = timed(lambda: job(n_job))

        def both():
            job(n_job)
            layer_steps()

        t_both = timed(both)
        assert layer.device_error() == 0
        out.append({"sm_margin": m, "layer_ms": round(t_layer, 3), "job_ms": round(t_job, 3),
                    "both_ms": round(t_both, 3), "job_launches": n_job,
                    "hidden": round((t_layer + t_job - t_both) / t_job, 3)})
        del layer
    print(json.dumps({"mode": "overlap_sweep", "workload": workload_name(cfg),
                      "steps": steps, "job": "1 GiB device-to-device copies on a second stream",
                      "results": out}), flush=True)


def bf16_host(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def per_kernel_table(cfg, per, kernel_ms, recompute, p_tc, p_bw):
    gf = gemm_flops(cfg, recompute)
    kb = kernel_bytes(cfg, recompute)
    out = {}
    for k, v in sorted(kernel_ms.items()):
        ent = {"ms": round(v, 4)}
        if k in gf:
            ent["tflops"] = round(gf[k] / (v / 1e3) / 1e12, 1)
            ent["frac_tensor"] = round(gf[k] / (v / 1e3) / 1e12 / p_tc, 3)
        if k in kb:
            ent["gbs"] = round(kb[k] / (v / 1e3) / 1e9, 1)
            ent["frac_hbm"] = round(kb[k] / (v / 1e3) / 1e9 / p_bw, 3)
        out[k] = ent
    return out


def dominant_roofline(cfg, per, kernel_ms, recompute, p_tc, p_bw, tc_kind, peak_src):
    """Roofline of the kernel with the largest share of the step: algorithmic flops or bytes
    per launch over its mean live duration, against the bound its arithmetic intensity sets."""
    gf = gemm_flops(cfg, recompute)
    kb = kernel_bytes(cfg, recompute)
    dom = max((k for k in kernel_ms if k in gf or k in kb), key=lambda k: sum(per[k]))
    dom_ms = kernel_ms[dom]
    t_tc = gf.get(dom, 0.0) / (p_tc * 1e12)
    t_bw = kb.get(dom, 0.0) / (p_bw * 1e9)
    if t_tc >= t_bw:
        bound, achieved, peak, unit = "tensor", gf[dom] / (dom_ms / 1e3) / 1e12, p_tc, "TFLOP/s"
        nominal = NOMINAL_TFLOPS[cfg.precision]
    else:
        bound, achieved, peak, unit = "hbm", kb[dom] / (dom_ms / 1e3) / 1e9, p_bw, "GB/s"
        nominal = NOMINAL_HBM_GBS
    return {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic_for(dom, cfg.name),
            "peak_kind": tc_kind if bound == "tensor" else f"hbm_gbs ({peak_src})",
            "frac_of_nominal": achieved / nominal, "nominal_peak": nominal,
            "flops_per_launch": gf.get(dom), "bytes_per_launch": kb.get(dom),
            "ms_per_launch": dom_ms}


def measure(cfg, args, world, local, steps, warmup, with_e2e):
    """Time `steps` layer steps (route + forward + backward) of workload `cfg` on this rank's
    GPU, after `warmup` untimed ones; per-kernel durations come from the library's launch
    timeline (CUDA events on the launching stream). Returns a dict of measurements."""
    import torch

    import grouped_gemm_device_gb300 as g

    dev = torch.device("cuda", local)
    t_gen = time.time()
    hin = host_inputs(cfg)
    t_gen = time.time() - t_gen
    desc = g.desc_from_config(cfg, sm_margin=args.sm_margin, recompute=args.recompute,
                              extras=args.extras)
    layer = g.MoELayer(desc, dev)
    fc1_bias = (torch.from_numpy(synth.gen_fc1_bias(cfg)).to(dev)
                if args.extras & g.EXTRA_BIAS else None)
    feat_scale = (torch.from_numpy(synth.gen_feat_scale(cfg)).to(dev)
                  if args.extras & g.EXTRA_SCALE else None)
    w1_log = torch.stack([bf16_host(w) for w in hin["w1"]]).to(dev)
    w1p = g.pack_w1(w1_log, gated=cfg.gated, ilv=cfg.ilv)
    del w1_log
    w2 = torch.stack([bf16_host(w) for w in hin["w2"]]).to(dev)
    logits = torch.from_numpy(hin["logits"]).to(dev)
    x = bf16_host(hin["x"]).to(dev)
    dy = bf16_host(hin["dy"]).to(dev)
    T = cfg.T

    def step():
        layer.route_permute(logits, x, T)
        layer.forward(w1p, w2, T, fc1_bias=fc1_bias, feat_scale=feat_scale)
        layer.backward(dy, w1p, w2, T, feat_scale=feat_scale)

    n_w = g.moe_launch_count()
    for _ in range(max(warmup, 1)):
        step()
    torch.cuda.synchronize()
    per_step_launches = (g.moe_launch_count() - n_w) // max(warmup, 1)
    assert layer.device_error() == 0, "device error during warm-up"

    tl = g.Timeline(min(8192, steps * per_step_launches + 16))
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    n0 = g.moe_launch_count()
    tl.begin()
    ev0.record()
    for _ in range(steps):
        step()
    ev1.record()
    torch.cuda.synchronize()
    n_rec = tl.end()
    launches = g.moe_launch_count() - n0
    barrier(world)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = ev0.elapsed_time(ev1) / steps
    ms_max = allreduce_max(ms, world)
    assert layer.device_error() == 0, "device error during timing"

    per = {}
    seen = {}
    for i, (name, dur) in enumerate(tl.durations(ev0)):
        if i % per_step_launches == 0:
            seen = {}
        j = seen.get(name, 0)
        seen[name] = j + 1
        per.setdefault(REPEATED[name][j] if name in REPEATED else name, []).append(dur)
    kernel_ms = {k: sum(v) / len(v) for k, v in per.items()}

    # the same steps with the forward reusing the block-scaled weight copies (gradient
    # accumulation over micro-batches): the step time without weight quantisation
    wq = None
    if cfg.precision != "bf16":
        layer.desc.reuse_weights = 1
        step()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k_r = max(3, steps // 2)
        e0.record()
        for _ in range(k_r):
            step()
        e1.record()
        torch.cuda.synchronize()
        layer.desc.reuse_weights = 0
        assert layer.device_error() == 0, "device error in the weight-reuse steps"
        ms_reuse = allreduce_max(e0.elapsed_time(e1) / k_r, world)
        wq = {"ms_per_step_with_weight_quant": ms_max,
              "ms_per_step_weights_reused": ms_reuse,
              "weight_quant_ms_in_step": sum(kernel_ms.get(k, 0.0) for k in WEIGHT_QUANT),
              "tflops_weights_reused": job_throughput(cfg.flops_fwd_bwd(), ms_reuse, world) / 1e12}

    # the step without the per-launch timeline, in ordinary stream order and with
    # programmatic dependent launch (each kernel's CTAs scheduled while the previous kernel's
    # last CTAs finish); the timeline's event after every launch would serialise the launches
    pdl = None
    if args.pdl_compare:
        k_p = max(5, steps // 2)
        times = {}
        for flag in (0, 1, 0, 1):
            layer.desc.pdl = flag
            step()
            torch.cuda.synchronize()
            barrier(world)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(k_p):
                step()
            e1.record()
            torch.cuda.synchronize()
            times.setdefault(flag, []).append(allreduce_max(e0.elapsed_time(e1) / k_p, world))
        layer.desc.pdl = 0
        assert layer.device_error() == 0, "device error in the launch-mode steps"
        pdl = {"ms_per_step_stream_order": min(times[0]), "ms_per_step_pdl": min(times[1]),
               "steps": k_p, "note": "no per-launch timeline; best of two runs each"}

    e2e = None
    if with_e2e:
        layer.desc.pdl = 1 if args.e2e_pdl else 0
        e2e = measure_e2e(cfg, layer, hin, logits, x, dy, w1p, w2, fc1_bias, feat_scale, world,
                          steps)
        e2e["pdl"] = bool(args.e2e_pdl)
        layer.desc.pdl = 0
    res = {"cfg": cfg, "ms": ms, "ms_max": ms_max, "per": per, "kernel_ms": kernel_ms,
           "launches": int(launches), "timeline_events": n_rec, "clocks": clocks, "wq": wq,
           "pdl": pdl,
           "e2e": e2e, "t_gen": t_gen, "ws_bytes": layer.ws_bytes, "hin": hin}
    del layer, w1p, w2, logits, x, dy
    torch.cuda.empty_cache()
    return res


def measure_e2e(cfg, layer, hin, logits, x, dy, w1p, w2, fc1_bias, feat_scale, world, steps):
    """End to end through the C ABI with host buffers: every step copies its inputs from pinned
    host memory and its results back, inside the timed region. The copies run on two side
    streams ordered by events so they overlap the layer's kernels: the next step's logits and
    x load once this step's routing has gathered x, dy loads during the forward, y returns
    during the backward, dx and d_probs during the next step."""
    import torch
    T = cfg.T
    flops = cfg.flops_fwd_bwd()
    h_logits = torch.from_numpy(hin["logits"]).pin_memory()
    h_x = bf16_host(hin["x"]).pin_memory()
    h_dy = bf16_host(hin["dy"]).pin_memory()
    h_y = torch.empty(T, cfg.H, dtype=torch.bfloat16).pin_memory()
    h_dx = torch.empty(T, cfg.H, dtype=torch.bfloat16).pin_memory()
    h_dp = torch.empty(T, cfg.k, dtype=torch.float32).pin_memory()
    main = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {n: torch.cuda.Event() for n in
          ("in", "routed", "dy", "fwd", "bwd", "y_out", "dx_out", "start")}

    def load_inputs():
        with torch.cuda.stream(h2d):
            logits.copy_(h_logits, non_blocking=True)
            x.copy_(h_x, non_blocking=True)
            ev["in"].record(h2d)

    def e2e_step():
        main.wait_event(ev["in"])
        layer.route_permute(logits, x, T)
        ev["routed"].record(main)
        with torch.cuda.stream(h2d):
            h2d.wait_event(ev["bwd"])       # the previous backward has read dy
            dy.copy_(h_dy, non_blocking=True)
            ev["dy"].record(h2d)
        load_inputs()                       # next step's inputs; x and logits are free
        main.wait_event(ev["y_out"])        # the previous y has left the device
        layer.forward(w1p, w2, T, fc1_bias=fc1_bias, feat_scale=feat_scale)
        ev["fwd"].record(main)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev["fwd"])
            h_y.copy_(layer.y[:T], non_blocking=True)
            ev["y_out"].record(d2h)
        main.wait_event(ev["dy"])
        main.wait_event(ev["dx_out"])       # the previous dx / d_probs have left
        layer.backward(dy, w1p, w2, T, feat_scale=feat_scale)
        ev["bwd"].record(main)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev["bwd"])
            h_dx.copy_(layer.dx[:T], non_blocking=True)
            h_dp.copy_(layer.d_probs[:T], non_blocking=True)
            ev["dx_out"].record(d2h)

    def e2e_run(n):
        for e in ("bwd", "y_out", "dx_out", "start"):
            ev[e].record(main)
        h2d.wait_event(ev["start"])
        load_inputs()
        for _ in range(n):
            e2e_step()
        main.wait_stream(h2d)
        main.wait_stream(d2h)

    e2e_run(3)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    k_e2e = max(10, steps // 4)
    e0.record()
    e2e_run(k_e2e)
    e1.record()
    torch.cuda.synchronize()
    ms_e2e = allreduce_max(e0.elapsed_time(e1) / k_e2e, world)
    bi = h_logits.numel() * 4 + h_x.numel() * 2 + h_dy.numel() * 2
    bo = h_y.numel() * 2 + h_dx.numel() * 2 + h_dp.numel() * 4
    return {"value": job_throughput(flops, ms_e2e, world) / 1e12, "unit": "TFLOPS",
            "ms_per_step": ms_e2e, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "tokens_per_s": T * world / (ms_e2e / 1e3)}


def summarise(r, args, world, peaks, peak_src):
    """The JSON fields of one measured workload."""
    cfg = r["cfg"]
    flops = cfg.flops_fwd_bwd()
    ms, ms_max = r["ms"], r["ms_max"]
    value = job_throughput(flops, ms_max, world) / 1e12
    p_tc, tc_kind = tensor_peak(peaks, cfg.precision, r["clocks"])
    p_bw = peaks.get("hbm_gbs", 6800.0)
    kb = kernel_bytes(cfg, args.recompute)
    gf = gemm_flops(cfg, args.recompute)
    step_bytes = sum(kb.values())
    step_ideal_ms = 1e3 * max(flops / (p_tc * 1e12), step_bytes / (p_bw * 1e9))
    gemm_total_ms = sum(r["kernel_ms"][k] for k in gf if k in r["kernel_ms"])
    out = {
        "workload": workload_name(cfg), "name": cfg.name, "ms_per_step": ms_max,
        "value": value, "unit": "TFLOPS", "tokens_per_s": cfg.T * world / (ms_max / 1e3),
        "dtype": DTYPE[cfg.precision], "flops_per_step": flops,
        "pct_tensor_peak": {"value": 100 * value / world / p_tc, "peak_tflops": p_tc,
                            "peak_kind": f"{tc_kind} ({peak_src})",
                            "pct_of_nominal": 100 * value / world /
                            NOMINAL_TFLOPS[cfg.precision],
                            "nominal_tflops": NOMINAL_TFLOPS[cfg.precision]},
        "step_roofline": {"ideal_ms": step_ideal_ms, "frac": step_ideal_ms / ms,
                          "bytes": step_bytes,
                          "bound": "tensor" if flops / (p_tc * 1e12) >=
                          step_bytes / (p_bw * 1e9) else "hbm"},
        "roofline": dominant_roofline(cfg, r["per"], r["kernel_ms"], args.recompute, p_tc, p_bw,
                                      tc_kind, peak_src),
        "kernels": per_kernel_table(cfg, r["per"], r["kernel_ms"], args.recompute, p_tc, p_bw),
        "gemm_share": gemm_total_ms / ms,
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if r["wq"]:
        out["weight_quant"] = r["wq"]
    if r["pdl"]:
        out["launch_mode"] = r["pdl"]
    return out


def maybe_spawn(args):
    """`--gpus N` (N > 1) outside torchrun starts N replica ranks under torch.distributed.run,
    so the line's n_gpus is the number of GPUs asked for; inside torchrun the world size must
    match the request."""
    ws = os.environ.get("WORLD_SIZE")
    if args.gpus > 1 and ws is None:
        import socket
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1", "--master-port",
               str(port), os.path.abspath(__file__), *sys.argv[1:]]
        os.execv(sys.executable, cmd)
    if ws is not None and int(ws) != args.gpus and args.gpus != 1:
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={ws}")


def extra_workloads(args):
    if args.workloads == "none" or args.tokens or args.experts or args.extras or args.recompute:
        return []
    if args.workloads == "auto":
        return list(EXTRA_WORKLOADS) if args.config == HEADLINE else []
    names = [n.strip() for n in args.workloads.split(",") if n.strip()]
    bad = [n for n in names if n not in synth.CONFIGS]
    if bad:
        sys.exit(f"bench.py: unknown workloads {bad}")
    return [n for n in names if n != args.config]


def main():
    args = parse()
    if args.overlap_sweep:
        overlap_sweep(args)
        return
    maybe_spawn(args)
    if args.impl == "reference":
        run_reference(args)
        return
    import torch

    import grouped_gemm_device_gb300 as g
    from grouped_gemm_device_gb300 import build as gbuild

    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    if rank == 0:
        gbuild.build()
    barrier(world)
    g.load()
    cfg = config_of(args)
    peaks, peak_src = load_peaks()

    r = measure(cfg, args, world, local, args.steps, args.warmup, not args.no_e2e)
    head = summarise(r, args, world, peaks, peak_src)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        # a bounded sample of about 10 s of host work: expert 0's routed tokens (up to 2048),
        # repeated until 10 s have passed (at most 8 passes)
        dt = fl = 0.0
        passes = 0
        while passes < 8 and (passes == 0 or dt < 10.0):
            d1, f1, sdesc, _ = oracle_sample(cfg, 2048, r["hin"])
            dt += d1
            fl += f1
            passes += 1
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOPS", "cores": blas_threads(),
               "host_cpu_count": HOST_CORES, "blas_threads": blas_threads(),
               "kind": "oracle", "sample": f"{passes} passes of: {sdesc}", "seconds": dt,
               "tokens_per_s_equiv": (fl / dt) / (cfg.flops_fwd_bwd() / cfg.T)}
    del r["hin"]

    others = []
    for name in extra_workloads(args):
        rw = measure(synth.CONFIGS[name], args, world, local, args.workload_steps, 3, False)
        del rw["hin"]
        others.append(summarise(rw, args, world, peaks, peak_src))

    if rank == 0:
        w_bytes = 2 * 2 * cfg.E * (cfg.N1 + cfg.F) * cfg.H
        line = {
            "metric": METRIC, "value": head["value"], "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE[cfg.precision],
            "data": "synthetic",
            "config": {"workload": workload_name(cfg), "parallelism": f"replicas x{world}",
                       "l2": f"no flush: each step streams {w_bytes / 1e9:.1f} GB of bf16 "
                             "weights and weight gradients, > 129 MB L2",
                       "sm_margin": args.sm_margin, "flops_per_step": cfg.flops_fwd_bwd(),
                       "recompute": bool(args.recompute), "extras": args.extras,
                       "workspace_bytes": r["ws_bytes"]},
            "tokens_per_s": head["tokens_per_s"],
            "pct_tensor_peak": head["pct_tensor_peak"],
            "step_roofline": head["step_roofline"],
            "gpu_launches": head["gpu_launches"],
            "roofline": head["roofline"],
            "kernels": head["kernels"],
            "gemm_share": head["gemm_share"],
            "timeline_events": r["timeline_events"],
            "e2e": r["e2e"],
            "cpu_baseline": cpu,
            "clocks": head["clocks"],
            "input_gen_s": round(r["t_gen"], 1),
        }
        if head.get("weight_quant"):
            line["weight_quant"] = head["weight_quant"]
        if head.get("launch_mode"):
            line["launch_mode"] = head["launch_mode"]
        if others:
            line["workloads"] = others
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
