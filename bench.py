#!/usr/bin/env python3
"""Benchmark of the blockwise-FP8 Transformer linear layer on B300.

One step is one training micro-step of a stack of blockwise-FP8 linear
layers: for every linear, forward (weight quantisation in 128x128 blocks,
activation quantisation in 1x128 groups along features and along tokens,
FPROP GEMM), then, in reverse order, backward (output-gradient quantisation
along features and along tokens, DGRAD and WGRAD GEMMs).  This is the linear
numerics of "Puro-2B: Poor Lab's Qwen2-1.5B Trained on RTX 5090 within
$5090", section 3.2, on synthetic inputs shaped like its layers (hidden 2048,
FFN 6144, 16 query + 8 KV heads of dim 128, 4 x 4096 tokens).

Arms
  default          the CUDA kernels behind libbfp8.so, inputs resident in HBM;
                   also reports
                     e2e           the same step through the public fused calls
                                   (linear_fwd / linear_bwd) with every input
                                   copied from pinned host memory and every
                                   weight gradient copied back, inside the
                                   timed region;
                     roofline      GEMM TFLOP/s against the FP8 tensor peak and
                                   quantiser GB/s against HBM bandwidth, from
                                   CUDA events around every call;
                     cpu_baseline  the CPU oracle timed on a bounded sample.
  --impl reference the CPU oracle on a bounded sample of the same workload
                   (this method has no other implementation to run).

The printed value is whole-job GEMM throughput: 2*M*N*K FLOPs of every FPROP,
DGRAD and WGRAD GEMM of the step, divided by the step time (quantisers
included).  Launch with N processes (torchrun) to run N independent replicas;
no data crosses between them.
"""

import argparse
import hashlib
import json
import os
import shutil
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "blockwise-FP8 GEMM TFLOP/s (fwd+dgrad+wgrad) and % of B300 FP8 dense peak"
UNIT = "TFLOP/s"

# Fallback denominators (one earlier B300 measurement), used only when the
# measured-peaks file is absent.
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
FP8_PER_BF16 = 4.5 / 2.25  # nominal dense FP8 : BF16 tensor rate on B300

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch,
# averaged over the launches of one stack layer (the same launches as every
# layer of the step: 24, or 21 with the batched weight quantiser), from an
# ncu capture of
#   python bench.py --layers 1 --steps 1 --warmup 0 --no-e2e --no-cpu-baseline
# Valid only for the kernel code whose hash (comments ignored) is the key;
# once the kernels change the bench line reports null until a new capture is
# recorded.
TRAFFIC = {
    "ad55d462807144a1": {"gemm": 232.3e6, "quant": 155.8e6},
    "1508b235cee025dc": {"gemm": 231.9e6, "quant": 155.5e6},
    # a layer's four weights in one batched launch: 21 launches per layer
    "e056ae426709bae9": {"gemm": 232.5e6, "quant": 213.2e6},
}


def strip_comments(src):
    """C/C++ source without // and /* */ comments and with whitespace
    collapsed, so that an edit of comments alone leaves the hash unchanged.
    String and character literals are kept verbatim."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash():
    """Hash of the kernel sources' code (comments and layout ignored)."""
    h = hashlib.sha256()
    for f in ("common.cuh", "gemm.cuh", "gemm_mx.cuh", "quant.cuh", "api.cu"):
        with open(os.path.join(ROOT, "blockwise_fp8_linear_quantise_b300", "csrc", f), encoding="utf-8") as fh:
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------- host logic
def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("b300", "reference"), default="b300")
    ap.add_argument("--workload", default="stack28",
                    choices=("tiny", "mlp_gateup", "mlp_down", "attn_proj", "stack28"))
    ap.add_argument("--layers", type=int, default=28, help="stack28 only: layers to run (profiling cases)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=4096)
    ap.add_argument("--ref-sample-tokens", type=int, default=1024)
    ap.add_argument("--scale-mode", choices=["amax448", "pow2", "mul_recip"], default="amax448",
                    help="group scale rule: amax/448 with codes of x/s (default), the power-of-two mode, or "
                         "amax/448 with codes of x * fp32(448/amax)")
    ap.add_argument("--main-grad", action="store_true",
                    help="WGRAD adds into fp32 main gradients (bfp8_fp8_block_gemm_accumulate) instead of bf16 dW")
    ap.add_argument("--cached-weights", action="store_true",
                    help="weights quantised once before the timed steps (cached across micro-steps)")
    ap.add_argument("--graph", action="store_true",
                    help="time the step as replays of a CUDA graph captured once (per-call rates from an eager pass)")
    ap.add_argument("--probe-swiglu", action="store_true",
                    help="time the SiLU-gated prologue (bfp8_swiglu_quantize_1x128) on the down projection's input")
    ap.add_argument("--probe-fp8-peak", action="store_true",
                    help="time the library FP8 GEMM (torch._scaled_mm, per-tensor scales, 8192^3) as a peak reference")
    ap.add_argument("--plan-configs", default="tiny,mlp_gateup,mlp_down,attn_proj,stack28",
                    help="--oracle-plan: the configurations to run, comma-separated")
    ap.add_argument("--oracle-plan", action="store_true",
                    help="time the CPU oracle on every configuration in full (stack28: layer 0 in full, 1/16 of the "
                         "output tiles of layers 1-27, extrapolated) against the GPU path, checking parity")
    ap.add_argument("--per-kernel", action="store_true",
                    help="time each ABI call of one stack layer alone: 10 warm-up calls, then the median of 50, "
                         "with L2 flushed (a 256 MB write) before every timed call")
    ap.add_argument("--probe-mx", action="store_true",
                    help="compare the MXFP8 1x32 recipe with the blockwise one on the mlp_down layer: accuracy of "
                         "every GEMM against the unquantised product, and time of quantisers and GEMMs")
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_group(world):
    """A gloo group for the barrier and the max over ranks (host tensors
    only: the replicas exchange no data)."""
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group("gloo")
    return dist.group.WORLD


def barrier(group):
    if group is not None:
        import torch.distributed as dist
        dist.barrier(group)


def max_over_ranks(x, group):
    if group is None:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def sum_over_ranks(x, group):
    if group is None:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return float(t.item())


def load_peaks():
    """(peaks, basis): the measured denominators, with 'sustained_sm_mhz', the
    median SM clock under load while the sustained bf16 peak was measured
    (None when the file does not record it)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        out = {k: float(d[k]) for k in FALLBACK_PEAKS}
        out["sustained_sm_mhz"] = (d.get("clocks_under_load") or {}).get("sm_mhz_median")
        return out, "measured"
    out = dict(FALLBACK_PEAKS)
    out["sustained_sm_mhz"] = None
    return out, "fallback"


def clock_normalised(achieved, peak, peak_mhz, run_mhz):
    """achieved / (peak scaled from the clock it was measured at to the run's
    median SM clock): a tensor-bound rate scales with the SM clock, so this
    compares the kernel and the peak at the same clock."""
    if not peak_mhz or not run_mhz:
        return None
    return round(achieved / (peak * run_mhz / peak_mhz), 4)


def linear_list(wl, layers):
    from blockwise_fp8_linear_quantise_b300 import workloads
    specs = []
    for s in wl.linears:
        li = workloads.layer_of(s)
        if li is None or li < layers:
            specs.append(s)
    return specs


def gemm_flops(specs):
    return sum(2 * s.M * s.N * s.K * (3 if s.backward else 1) for s in specs)


def workload_config(wl, specs, layers, scale_mode="amax448", main_grad=False, cached_weights=False, graph=False):
    cfg = {"workload": wl.name, "linears": len(specs), "tokens": specs[0].M, "scale_mode": scale_mode,
           "launch": "CUDA-graph replay" if graph else "eager ABI calls",
           "dW": "fp32 main-grad accumulate" if main_grad else "bf16",
           "weights": "quantised once (cached)" if cached_weights else "quantised every step",
           "shapes_MNK": sorted({(s.M, s.N, s.K) for s in specs}),
           "passes": "fprop+dgrad+wgrad" if specs[0].backward else "fprop",
           "l2": "inputs larger than L2: each step streams several GB through HBM (no explicit flush)",
           "parallelism": "replicas (one independent step per GPU)"}
    if wl.name == "stack28":
        cfg["layers"] = layers
        cfg["what"] = ("Puro-2B linear stack, one micro-step: per layer QKV 2048->4096, O 2048->2048, "
                       "gate+up 2048->12288, down 6144->2048 on 16384 tokens; activations and output gradients "
                       "N(0,1) with 0.1% x50 outliers, weights N(0,0.02^2), distinct per layer")
    return cfg


def summarise_clocks(rows):
    """rows: parsed nvidia-smi samples -> the clocks object of the JSON line."""
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    sm = [r["sm"] for r in rows if r["sm"] is not None]
    reasons = set()
    for r in rows:
        reasons.update(r["active"])
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(r["sm_max"] for r in rows if r["sm_max"] is not None) if sm else None,
            "power_w_max": max((r["power"] for r in rows if r["power"] is not None), default=None),
            "reasons": sorted(reasons), "samples": len(rows)}


class ClockSampler:
    """nvidia-smi sampling of SM clock, power and throttle reasons while the
    timed region runs."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        exe = shutil.which("nvidia-smi")
        if exe is None or self.gpu_id is None:
            return
        self.proc = subprocess.Popen(
            [exe, "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
             "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)

    def stop(self):
        if self.proc is None:
            return summarise_clocks([])
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue

            def num(v):
                try:
                    return float(v)
                except ValueError:
                    return None
            rows.append({"sm": num(parts[0]), "sm_max": num(parts[1]), "power": num(parts[2]),
                         "active": [n for n, v in zip(self.NAMES, parts[3:]) if v.lower() == "active"]})
        return summarise_clocks(rows)


def cpu_model():
    """The host CPU's model name (Linux /proc/cpuinfo), or None."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def host_info():
    from oracle import parallel
    return {"nproc": os.cpu_count(), "usable_cpus": parallel.workers(), "cpu_model": cpu_model()}


# ------------------------------------------------------------ oracle timing
def oracle_sample(wl, specs, tokens):
    """CPU inputs for a bounded oracle sample: the first `tokens` tokens of
    every distinct linear shape of the workload's first layer, drawn from the
    workload's own distributions."""
    from blockwise_fp8_linear_quantise_b300 import workloads
    seen, sample = set(), []
    for s in specs:
        key = (s.N, s.K, s.backward)
        if key in seen:
            continue
        seen.add(key)
        m = min(tokens, s.M)
        f = lambda tag, shape: workloads.to_bf16(
            workloads.draw(wl.dists[tag], shape, wl.seed, tag + "#cpu-sample")).float().numpy()
        x = f(s.x_tag, (m, s.K))
        w = f(s.w_tag, (s.N, s.K))
        dy = f(s.dy_tag, (m, s.N)) if s.backward else None
        sample.append((x, w, dy))
    return sample


def run_oracle(sample, scale_mode="amax448"):
    """Oracle linear forward (+ backward) over the sample, its GEMMs spread
    over every host core by blocks of output rows (bit-identical to the
    serial oracle); returns GEMM FLOPs."""
    from oracle import parallel
    flops = 0
    for x, w, dy in sample:
        _, saved = parallel.linear_fwd(x, w, scale_mode=scale_mode)
        flops += 2 * x.shape[0] * w.shape[0] * x.shape[1]
        if dy is not None:
            parallel.linear_bwd(dy, saved, scale_mode=scale_mode)
            flops += 4 * x.shape[0] * w.shape[0] * x.shape[1]
    return flops


def oracle_cores():
    from oracle import parallel
    parallel.pool()  # started (spawn) before the timing
    return parallel.workers()


def describe_sample(sample):
    return "; ".join(f"M={x.shape[0]} N={w.shape[0]} K={x.shape[1]} {'fwd+bwd' if dy is not None else 'fwd'}"
                     for x, w, dy in sample)


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from blockwise_fp8_linear_quantise_b300 import workloads
    wl = workloads.make(args.workload)
    specs = linear_list(wl, args.layers)
    sample = oracle_sample(wl, specs, args.ref_sample_tokens)
    cores = oracle_cores()
    for _ in range(args.warmup):
        run_oracle(sample, args.scale_mode)
    t0 = time.perf_counter()
    flops = 0
    for _ in range(args.steps):
        flops += run_oracle(sample, args.scale_mode)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64/f32 (CPU oracle)",
            "data": "synthetic", "config": workload_config(wl, specs, args.layers, args.scale_mode),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "per step: " + describe_sample(sample)
                                       + " (quantisers and GEMMs split over a spawn process pool)",
                             **host_info()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------- GPU runner
class StackRunner:
    """Device buffers and the per-step call sequence of a workload.

    The step is issued as the C ABI's component calls (the same kernels, in
    the same order, as bfp8_linear_fwd / bfp8_linear_bwd) so that CUDA events
    can separate the quantiser and GEMM time.  Arguments are marshalled once;
    a step only makes the ctypes calls.
    """

    def __init__(self, wl, specs, dev, scale_mode="amax448", main_grad=False, cached_weights=False):
        import torch
        from blockwise_fp8_linear_quantise_b300 import _lib, ops, workloads
        self.torch = torch
        self.lib = _lib.load()
        self.ops = ops
        self.scale_mode = scale_mode
        self.mode_id = ops.SCALE_MODES[scale_mode]
        self.main_grad = main_grad            # WGRAD adds into fp32 main gradients
        self.cached_weights = cached_weights  # weights quantised once, before any step
        self.specs = specs
        self.dev = dev
        u8, f32, bf16 = torch.uint8, torch.float32, torch.bfloat16
        E = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)

        # inputs
        self.inputs = {}
        device_draw = wl.name == "stack28"
        for s in specs:
            li = workloads.layer_of(s)
            for tag, layer in ((s.x_tag, None), (s.w_tag, li), (s.dy_tag if s.backward else None, None)):
                if tag is None or (tag, layer) in self.inputs:
                    continue
                t = (workloads.tensor_cuda(wl, tag, layer, device=dev) if device_draw
                     else workloads.tensor(wl, tag, layer).to(dev))
                self.inputs[(tag, layer)] = t.contiguous()

        # scratch per shape, saved tensors and weight gradients per linear
        self.scratch = {}
        self.saved, self.dW = [], []
        ws = 0
        for s in specs:
            M, N, K = s.M, s.N, s.K
            key = (M, N, K)
            if key not in self.scratch:
                self.scratch[key] = dict(Xq=E((M, K), u8), sX=E((K // 128, M), f32),
                                         Y=E((M, N), bf16), dYq=E((M, N), u8), sdY=E((N // 128, M), f32),
                                         dYqT=E((N, M), u8), sdYT=E((M // 128, N), f32), dX=E((M, K), bf16))
            self.saved.append(dict(WqT=E((K, N), u8), sW=E((N // 128, K // 128), f32),
                                   XqT=E((K, M), u8), sXT=E((M // 128, K), f32)))
            if cached_weights:
                self.saved[-1]["Wq"] = E((N, K), u8)
            if s.backward:
                self.dW.append(torch.zeros((N, K), dtype=f32, device=dev) if main_grad else E((N, K), bf16))
            else:
                self.dW.append(None)
            ws = max(ws, ops.gemm_workspace_bytes(ops.FPROP, M, N, K))
            if s.backward:
                ws = max(ws, ops.gemm_workspace_bytes(ops.DGRAD, M, K, N),
                         ops.gemm_workspace_bytes(ops.WGRAD, N, K, M),
                         ops.linear_bwd_workspace_bytes(M, N, K))
            ws = max(ws, ops.linear_fwd_workspace_bytes(M, N, K))
        self.ws = E((max(ws, 256),), u8)
        self.ws_bytes = self.ws.numel()
        if cached_weights:  # once per optimizer step, outside the timed micro-steps
            for i, s in enumerate(specs):
                sv = self.saved[i]
                ops.quantize_w_128x128(self.inputs[(s.w_tag, workloads.layer_of(s))], q=sv["Wq"], qT=sv["WqT"],
                                       s=sv["sW"], scale_mode=scale_mode)
        self._marshal()

    def _marshal(self):
        """Argument tuples of every ABI call of one step, with their kind and
        algorithmic work (FLOPs for GEMMs, bytes for quantisers)."""
        P = lambda t: None if t is None else t.data_ptr()
        lib = self.lib
        from blockwise_fp8_linear_quantise_b300 import _lib, workloads
        fwd, bwd = [], []
        # A layer's weights are quantised by one batched call before its first
        # linear; the fprop codes of a layer's weights go to per-position
        # scratch so that no two of them share a buffer.
        layer_specs = {}
        for i, s in enumerate(self.specs):
            layer_specs.setdefault(workloads.layer_of(s), []).append(i)
        wq_scratch = {}
        wq_of = {}
        for li, idx in layer_specs.items():
            for pos, i in enumerate(idx):
                s = self.specs[i]
                key = (pos, s.N, s.K)
                if key not in wq_scratch:
                    wq_scratch[key] = self.torch.empty((s.N, s.K), dtype=self.torch.uint8, device=self.dev)
                wq_of[i] = wq_scratch[key]
        self._wq_scratch, self._jobs = wq_scratch, []
        for i, s in enumerate(self.specs):
            M, N, K = s.M, s.N, s.K
            sc, sv = self.scratch[(M, N, K)], self.saved[i]
            X = self.inputs[(s.x_tag, None)]
            ne_x = M * K
            Wq = sv["Wq"] if self.cached_weights else wq_of[i]
            idx = layer_specs[workloads.layer_of(s)]
            if not self.cached_weights and idx[0] == i:
                jobs = (_lib.WJob * len(idx))()
                ne_w = 0
                for k, j in enumerate(idx):
                    sj, svj = self.specs[j], self.saved[j]
                    Wj = self.inputs[(sj.w_tag, workloads.layer_of(sj))]
                    jobs[k] = _lib.WJob(P(Wj), sj.N, sj.K, P(wq_of[j]), P(svj["WqT"]), P(svj["sW"]))
                    ne_w += sj.N * sj.K
                self._jobs.append(jobs)
                fwd.append(("quant_w", ne_w * (4 + 4 / 16384), lib.bfp8_quantize_w_128x128_batch,
                            (jobs, len(idx), self.mode_id)))
            fwd.append(("quant_act", ne_x * (4 + 8 / 128), lib.bfp8_quantize_act_1x128_ex,
                        (P(X), M, K, P(sc["Xq"]), P(sc["sX"]), P(sv["XqT"]), P(sv["sXT"]), self.mode_id)))
            fwd.append(("fprop", 2.0 * M * N * K, lib.bfp8_fp8_block_gemm,
                        (self.ops.FPROP, P(sc["Xq"]), P(sc["sX"]), P(Wq), P(sv["sW"]), M, N, K, P(sc["Y"]),
                         None, None, P(self.ws), self.ws_bytes)))
            if s.backward:
                dY = self.inputs[(s.dy_tag, None)]
                ne_y = M * N
                b = [("quant_act", ne_y * (4 + 8 / 128), lib.bfp8_quantize_act_1x128_ex,
                      (P(dY), M, N, P(sc["dYq"]), P(sc["sdY"]), P(sc["dYqT"]), P(sc["sdYT"]), self.mode_id)),
                     ("dgrad", 2.0 * M * N * K, lib.bfp8_fp8_block_gemm,
                      (self.ops.DGRAD, P(sc["dYq"]), P(sc["sdY"]), P(sv["WqT"]), P(sv["sW"]), M, K, N, P(sc["dX"]),
                       None, None, P(self.ws), self.ws_bytes)),
                     ("wgrad", 2.0 * M * N * K, lib.bfp8_fp8_block_gemm_accumulate,
                      (self.ops.WGRAD, P(sc["dYqT"]), P(sc["sdYT"]), P(sv["XqT"]), P(sv["sXT"]), N, K, M,
                       P(self.dW[i]), P(self.ws), self.ws_bytes)) if self.main_grad else
                     ("wgrad", 2.0 * M * N * K, lib.bfp8_fp8_block_gemm,
                      (self.ops.WGRAD, P(sc["dYqT"]), P(sc["sdYT"]), P(sv["XqT"]), P(sv["sXT"]), N, K, M,
                       P(self.dW[i]), None, None, P(self.ws), self.ws_bytes))]
                bwd.append(b)
        self.calls = fwd + [c for b in reversed(bwd) for c in b]

    def step(self, marks=None):
        """One micro-step on the current stream.  With `marks`, records a
        CUDA event after every call: marks gets [(event, kind, work), ...]
        starting with (event, None, 0)."""
        torch = self.torch
        stream = torch.cuda.current_stream().cuda_stream
        if marks is not None:
            e = torch.cuda.Event(enable_timing=True)
            e.record()
            marks.append((e, None, 0))
        for kind, work, fn, args in self.calls:
            st = fn(*args, stream)
            if st != 0:
                raise RuntimeError(f"{kind}: status {st}")
            if marks is not None:
                e = torch.cuda.Event(enable_timing=True)
                e.record()
                marks.append((e, kind, work))

    # ------------------------------------------------------------ e2e arm
    def e2e_setup(self):
        """Pinned host copies of every input, a second device copy of the
        inputs (so that a step's inputs can be uploaded while the previous step
        computes), pinned host buffers for the weight gradients."""
        torch = self.torch
        self.h_inputs = {k: v.cpu().pin_memory() for k, v in self.inputs.items()}
        self.d_sets = [self.inputs, {k: torch.empty_like(v) for k, v in self.inputs.items()}]
        self.h_dW = [None if d is None else torch.empty(d.shape, dtype=d.dtype, pin_memory=True) for d in self.dW]
        # forward-only linears read back their outputs instead
        self.h_out = [None if s.backward else torch.empty((s.M, s.N), dtype=torch.bfloat16, pin_memory=True)
                      for s in self.specs]
        self.h2d_bytes = sum(v.numel() * v.element_size() for v in self.h_inputs.values())
        self.d2h_bytes = (sum(d.numel() * d.element_size() for d in self.dW if d is not None) +
                          sum(h.numel() * h.element_size() for h in self.h_out if h is not None))
        # upload order of one step: the forward's inputs in layer order, then
        # the output gradients in the order the backward uses them
        from blockwise_fp8_linear_quantise_b300 import workloads
        order = []
        for s in self.specs:
            for key in ((s.x_tag, None), (s.w_tag, workloads.layer_of(s))):
                if key not in order:
                    order.append(key)
        for s in reversed(self.specs):
            if s.backward and (s.dy_tag, None) not in order:
                order.append((s.dy_tag, None))
        self.upload_order = order

    def e2e_run(self, steps):
        """`steps` end-to-end steps on the current stream: host inputs ->
        device, the fused public calls, weight gradients -> host.

        Copies run on their own streams and overlap the kernels.  Step i's
        inputs go to device copy i % 2: step 0's are uploaded first, and step
        i + 1's are uploaded while step i computes, once step i - 1 has
        finished with that copy.  Each weight gradient is read back as soon as
        its WGRAD is done.  Every step's uploads and read-backs happen inside
        the call, which returns once the last read-back is complete."""
        torch, ops = self.torch, self.ops
        from blockwise_fp8_linear_quantise_b300 import workloads
        ms = torch.cuda.current_stream()
        if not hasattr(self, "_up"):
            self._up, self._down = torch.cuda.Stream(), torch.cuda.Stream()
        up, down = self._up, self._down
        start = torch.cuda.Event()
        start.record(ms)
        up.wait_event(start)
        down.wait_event(start)
        set_free = [start, start]  # compute finished with device copy k
        dw_read = {}               # weight gradient j read back (previous step)

        def upload(k):
            """Uploads one step's inputs into device copy k; returns their events."""
            evs = {}
            up.wait_event(set_free[k])
            with torch.cuda.stream(up):
                for key in self.upload_order:
                    self.d_sets[k][key].copy_(self.h_inputs[key], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(up)
                    evs[key] = ev
            return evs

        pending = upload(0)
        for i in range(steps):
            k = i % 2
            inputs, evs = self.d_sets[k], pending
            if i + 1 < steps:
                pending = upload(1 - k)
            for j, s in enumerate(self.specs):
                keys = [(s.x_tag, None), (s.w_tag, workloads.layer_of(s))]
                for key in keys:
                    ms.wait_event(evs[key])
                Y = self.scratch[(s.M, s.N, s.K)]["Y"]
                ops.linear_fwd(inputs[keys[0]], inputs[keys[1]], Y=Y, saved=self.saved[j], workspace=self.ws,
                               scale_mode=self.scale_mode)
                if not s.backward:
                    done = torch.cuda.Event()
                    done.record(ms)
                    down.wait_event(done)
                    with torch.cuda.stream(down):
                        self.h_out[j].copy_(Y, non_blocking=True)
                    # the next step's forward writes Y again only after this read
                    rd = torch.cuda.Event()
                    rd.record(down)
                    ms.wait_event(rd)
            for j in reversed(range(len(self.specs))):
                s = self.specs[j]
                if not s.backward:
                    continue
                ms.wait_event(evs[(s.dy_tag, None)])
                if j in dw_read:
                    ms.wait_event(dw_read[j])  # the previous step's read-back of dW[j] is done
                dX = self.scratch[(s.M, s.N, s.K)]["dX"]
                ops.linear_bwd(inputs[(s.dy_tag, None)], self.saved[j], dX=dX, dW=self.dW[j], workspace=self.ws,
                               scale_mode=self.scale_mode)
                done = torch.cuda.Event()
                done.record(ms)
                down.wait_event(done)
                with torch.cuda.stream(down):
                    self.h_dW[j].copy_(self.dW[j], non_blocking=True)
                    rd = torch.cuda.Event()
                    rd.record(down)
                dw_read[j] = rd
            fin = torch.cuda.Event()
            fin.record(ms)
            set_free[k] = fin
        end = torch.cuda.Event()
        end.record(down)
        ms.wait_event(end)
        ms.wait_event(set_free[(steps - 1) % 2])


def interval_stats(marks):
    """Sum of event intervals per kind: {kind: [launch_calls, ms, work]}."""
    out = {}
    prev = None
    for e, kind, work in marks:
        if kind is not None and prev is not None:
            ms = prev.elapsed_time(e)
            d = out.setdefault(kind, [0, 0.0, 0.0])
            d[0] += 1
            d[1] += ms
            d[2] += work
        prev = e
    return out


def gpu_uuid(dev):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


def gpu_arm(args):
    import torch
    rank, world, local = dist_env()
    group = init_group(world)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the kernels need an sm_103a GPU; there is no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from blockwise_fp8_linear_quantise_b300 import build as bld, ops, workloads
    bld.build()
    wl = workloads.make(args.workload)
    layers = args.layers if args.workload == "stack28" else 0
    specs = linear_list(wl, layers)
    runner = StackRunner(wl, specs, dev, args.scale_mode, args.main_grad, args.cached_weights)
    flops_step = gemm_flops(specs)

    # warm-up
    for _ in range(args.warmup):
        runner.step()
    torch.cuda.synchronize()
    if ops.sync_status() != 0:
        raise SystemExit("device status not ok after warm-up")

    # --graph: the step's calls are captured once into a CUDA graph, and the
    # timed region replays it (no host work per launch)
    graph = None
    if args.graph:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            runner.step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        n0 = ops.launch_count()
        with torch.cuda.graph(graph):
            runner.step()
        graph_launches = ops.launch_count() - n0
        graph.replay()
        torch.cuda.synchronize()

    # timed region
    clocks = ClockSampler(gpu_uuid(dev))
    barrier(group)
    torch.cuda.synchronize()
    clocks.start()
    launches0 = ops.launch_count()
    marks = []
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            runner.step(marks)
    t_end.record()
    torch.cuda.synchronize()
    launches = ops.launch_count() - launches0 if graph is None else graph_launches * args.steps
    clk = clocks.stop()
    barrier(group)
    st = ops.sync_status()
    if st != 0:
        raise SystemExit(f"device status {st} in the timed region")
    if graph is not None:
        # per-call durations come from an eager pass of the same steps
        for _ in range(args.steps):
            runner.step(marks)
        torch.cuda.synchronize()
    ms_local = t_start.elapsed_time(t_end)
    ms = max_over_ranks(ms_local, group)
    total_flops = sum_over_ranks(flops_step * args.steps, group)
    value = total_flops / (ms * 1e-3) / 1e12
    ms_per_step = ms / args.steps

    stats = interval_stats(marks)
    peaks, basis = load_peaks()
    fp8_sust = peaks["bf16_tflops_sustained"] * FP8_PER_BF16
    fp8_burst = peaks["bf16_tflops"] * FP8_PER_BF16
    g = [stats[k] for k in ("fprop", "dgrad", "wgrad") if k in stats]
    g_calls = sum(x[0] for x in g)
    g_ms = sum(x[1] for x in g)
    g_flops = sum(x[2] for x in g)
    g_achieved = g_flops / (g_ms * 1e-3) / 1e12
    q = [stats[k] for k in ("quant_w", "quant_act") if k in stats]
    q_ms = sum(x[1] for x in q)
    q_bytes = sum(x[2] for x in q)
    q_achieved = q_bytes / (q_ms * 1e-3) / 1e9 if q_ms > 0 else None
    total_ms = sum(v[1] for v in stats.values())
    src_hash = kernel_source_hash()
    # the record is of the default step: amax/448 scales, bf16 dW, weights quantised per use
    default_step = args.scale_mode == "amax448" and not args.main_grad and not args.cached_weights
    rec = TRAFFIC.get(src_hash, {}) if args.workload == "stack28" and default_step else {}
    traffic = rec.get("gemm")
    per_kernel = {k: {"calls": v[0], "ms_total": round(v[1], 3), "share": round(v[1] / total_ms, 4),
                      ("TFLOP/s" if k in ("fprop", "dgrad", "wgrad") else "GB/s"):
                          round(v[2] / (v[1] * 1e-3) / (1e12 if k in ("fprop", "dgrad", "wgrad") else 1e9), 1)}
                  for k, v in sorted(stats.items())}
    roofline = {"bound": "tensor", "kernel": "block_gemm_kernel (+ split-K reduce where planned), all GEMM calls",
                "achieved": round(g_achieved, 1), "peak": round(fp8_sust, 1), "unit": "TFLOP/s",
                "frac": round(g_achieved / fp8_sust, 4),
                "peak_basis": f"{FP8_PER_BF16:g} x {basis} bf16 sustained ({peaks['bf16_tflops_sustained']}) TFLOP/s",
                "frac_of_burst": round(g_achieved / fp8_burst, 4),
                "frac_clock_normalised": clock_normalised(g_achieved, fp8_sust, peaks["sustained_sm_mhz"],
                                                          clk.get("sm_mhz")),
                "clock_basis": f"sustained peak measured at a median {peaks['sustained_sm_mhz']} MHz, scaled to this "
                               f"run's median {clk.get('sm_mhz')} MHz",
                "traffic": traffic, "flops_per_call": round(g_flops / max(g_calls, 1))}
    roofline_q = None
    if q_achieved is not None:
        roofline_q = {"bound": "hbm", "kernel": "quantize_tile_kernel (activation dual + weight)",
                      "achieved": round(q_achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                      "frac": round(q_achieved / peaks["hbm_gbs"], 4), "peak_basis": f"{basis} HBM copy",
                      "frac_clock_normalised": round(q_achieved / peaks["hbm_gbs"], 4),
                      "clock_basis": "HBM bandwidth does not scale with the SM clock: the same as frac",
                      "bytes_per_call": round(q_bytes / max(sum(x[0] for x in q), 1)), "traffic": rec.get("quant")}

    # e2e through the public fused calls with host buffers
    e2e = None
    if args.main_grad or args.cached_weights:
        e2e = {"value": None, "unit": UNIT,
               "skipped": "measured for the default step only (fused linear_fwd / linear_bwd with bf16 dW)"}
    elif not args.no_e2e:
        runner.e2e_setup()
        runner.e2e_run(max(1, min(args.warmup, 2)))
        torch.cuda.synchronize()
        barrier(group)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        e2e_steps = max(1, args.steps)  # as many steps as the device-timed region
        runner.e2e_run(e2e_steps)
        b.record()
        torch.cuda.synchronize()
        barrier(group)
        if ops.sync_status() != 0:
            raise SystemExit("device status not ok in the e2e region")
        ems = max_over_ranks(a.elapsed_time(b), group)
        eflops = sum_over_ranks(flops_step * e2e_steps, group)
        e2e = {"value": eflops / (ems * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": runner.h2d_bytes,
               "d2h_bytes_per_step": runner.d2h_bytes, "ms_per_step": ems / e2e_steps, "steps": e2e_steps,
               "calls": "linear_fwd / linear_bwd (fused public calls); every step's inputs uploaded from pinned host "
                        "memory and every weight gradient read back, on copy streams overlapping the kernels (the "
                        "next step's inputs go up into a second device copy while a step computes)"}

    # CPU oracle on a bounded sample (rank 0, single GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = oracle_sample(wl, specs, args.cpu_sample_tokens)
        cores = oracle_cores()
        t0 = time.perf_counter()
        f = run_oracle(sample, args.scale_mode)
        dt = time.perf_counter() - t0
        cpu = {"value": f / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": describe_sample(sample) + f" ({dt:.1f} s; quantisers and GEMMs split over a spawn "
                                                   f"process pool of {cores})",
               **host_info()}

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate, bf16 out)",
                "data": "synthetic", "config": workload_config(wl, specs, layers, args.scale_mode, args.main_grad, args.cached_weights,
                                          args.graph),
                "roofline": roofline, "roofline_quant": roofline_q, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches, "clocks": clk, "per_kernel": per_kernel,
                "gemm_tflop_per_step": flops_step / 1e12, "kernel_source": src_hash}
        print(json.dumps(line), flush=True)
    if group is not None:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def fp8_peak_probe():
    """Dense FP8 GEMM throughput of the vendor library on this GPU: 8192^3
    E4M3 x E4M3 with per-tensor scales, bf16 out.  Best of 10 (burst) and a
    4-second back-to-back loop (sustained), with the clocks seen meanwhile."""
    import torch
    n = 8192
    dev = torch.device("cuda")
    a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()
    one = torch.ones((), device=dev)
    mm = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    for _ in range(3):
        mm()
    torch.cuda.synchronize()
    best = 1e30
    for _ in range(10):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        mm()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    clocks = ClockSampler(gpu_uuid(dev))
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    reps = 0
    e0.record()
    while time.perf_counter() - t0 < 4.0:
        for _ in range(20):
            mm()
        reps += 20
        torch.cuda.synchronize()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    flop = 2.0 * n ** 3
    line = {"probe": "fp8_dense_peak", "how": "torch._scaled_mm e4m3 8192^3 per-tensor scales, bf16 out",
            "burst_tflops": flop / (best * 1e-3) / 1e12,
            "sustained_tflops": flop * reps / (e0.elapsed_time(e1) * 1e-3) / 1e12, "clocks": clk}
    print(json.dumps(line), flush=True)
    return 0


def oracle_plan(args):
    """The oracle timing plan: the CPU oracle, on every host core, against the
    GPU path on the same CPU-drawn inputs of every configuration.

    tiny, mlp_gateup, mlp_down, attn_proj: every quantisation and every GEMM
    of the configuration in full.  stack28: every layer's quantisations in
    full; layer 0's GEMMs in full; for layers 1-27 a seeded sample of 1/16 of
    each GEMM's 128 x 128 output tiles (a quarter of the 128-row blocks times
    a quarter of the 128-column blocks), whose oracle time is extrapolated to
    the whole GEMM and labelled so.  Parity is checked wherever the oracle ran:
    codes and scales bit for bit, GEMM bf16 outputs within relative Frobenius
    error 1e-3.  One JSON line per configuration."""
    import numpy as np
    import torch
    from blockwise_fp8_linear_quantise_b300 import ops, workloads
    from oracle import parallel
    cores = oracle_cores()
    host = host_info()
    np32 = lambda t: t.float().cpu().numpy()
    u8 = lambda t: t.cpu().numpy()

    def same(got, want, what):
        g, w = np.asarray(got), np.asarray(want)
        if g.dtype == np.float32:
            g, w = g.view(np.uint32), w.view(np.uint32)
        if not np.array_equal(g, w):
            raise SystemExit(f"oracle plan: {what} differs from the oracle")

    def rel(g, w):
        w = np.asarray(w, np.float64)
        return float(np.linalg.norm(np.asarray(g, np.float64) - w) / max(np.linalg.norm(w), 1e-300))

    gpu_q = {}

    def quant(kind, t, key):
        """GPU and oracle quantisation of one tensor; returns the oracle's outputs."""
        if key in gpu_q:
            return gpu_q[key]
        x = t.to("cuda")
        t0 = time.perf_counter()
        if kind == "w":
            o = parallel.quantize_w_128x128(np32(t))
            g = ops.quantize_w_128x128(x)
            nbytes = t.numel() * (4 + 4 / 16384)
        else:
            o = parallel.quantize_act_1x128(np32(t)) + parallel.quantize_act_tokens_1x128(np32(t))
            g = ops.quantize_act_1x128(x, rows=True, tokens=True)
            nbytes = t.numel() * (4 + 8 / 128)
        dt = time.perf_counter() - t0
        assert ops.sync_status() == 0
        for gi, oi, nm in zip(g, o, ("q", "s", "qT", "sT") if kind != "w" else ("Wq", "WqT", "sW")):
            same(u8(gi), oi, f"{key} {nm}")
        stats["quant_s"] += dt
        stats["quant_bytes"] += nbytes
        gpu_q[key] = (g, o)
        return g, o

    rng = np.random.default_rng(2024)
    for name in args.plan_configs.split(","):
        wl = workloads.make(name)
        gpu_q.clear()
        stats = {"quant_s": 0.0, "quant_bytes": 0.0, "gemm_s_full": 0.0, "gemm_flop_full": 0.0,
                 "gemm_s_sampled": 0.0, "gemm_flop_sampled": 0.0, "gemm_s_extrapolated": 0.0, "worst_rel_fro": 0.0,
                 "gemms_full": 0, "gemms_sampled": 0}
        cache = {}
        tens = lambda tag, layer=None: cache.setdefault((tag, layer), workloads.tensor(wl, tag, layer))
        for s in wl.linears:
            li = workloads.layer_of(s)
            sampled = name == "stack28" and li > 0
            (Xq, sX, XqT, sXT), (oXq, osX, oXqT, osXT) = quant("a", tens(s.x_tag), s.x_tag)
            (Wq, WqT, sW), (oWq, oWqT, osW) = quant("w", tens(s.w_tag, li), f"{s.w_tag}@{li}")
            gemms = [("fprop", ops.FPROP, (Xq, sX, Wq, sW), (oXq, osX, oWq, osW), s.M, s.N, s.K)]
            if s.backward:
                (dYq, sdY, dYqT, sdYT), (odYq, osdY, odYqT, osdYT) = quant("a", tens(s.dy_tag), s.dy_tag)
                gemms += [("dgrad", ops.DGRAD, (dYq, sdY, WqT, sW), (odYq, osdY, oWqT, osW), s.M, s.K, s.N),
                          ("wgrad", ops.WGRAD, (dYqT, sdYT, XqT, sXT), (odYqT, osdYT, oXqT, osXT), s.N, s.K, s.M)]
            for gname, lay, gargs, oargs, M, N, K in gemms:
                Cg = ops.fp8_block_gemm(lay, *gargs)
                assert ops.sync_status() == 0
                rows = cols = None
                if sampled:
                    rb = np.sort(rng.choice(M // 128, max(1, M // 512), replace=False))
                    cb = np.sort(rng.choice(N // 128, max(1, N // 512), replace=False))
                    rows = (rb[:, None] * 128 + np.arange(128)).ravel()
                    cols = (cb[:, None] * 128 + np.arange(128)).ravel()
                    Cg = Cg[torch.as_tensor(rows, device=Cg.device)][:, torch.as_tensor(cols, device=Cg.device)]
                got = np32(Cg)
                del Cg
                t0 = time.perf_counter()
                _, want = parallel.gemm_rows(gname, *oargs, rows=rows, cols=cols)
                dt = time.perf_counter() - t0
                err = rel(got, want)
                if not err <= 1e-3:
                    raise SystemExit(f"oracle plan: {name} {s.name} {gname} relative Frobenius error {err:.3e}")
                stats["worst_rel_fro"] = max(stats["worst_rel_fro"], err)
                flop = 2.0 * M * N * K
                if rows is None:
                    stats["gemm_s_full"] += dt
                    stats["gemm_flop_full"] += flop
                    stats["gemms_full"] += 1
                else:
                    frac = len(rows) * len(cols) / (M * N)
                    stats["gemm_s_sampled"] += dt
                    stats["gemm_flop_sampled"] += flop * frac
                    stats["gemm_s_extrapolated"] += dt / frac
                    stats["gemms_sampled"] += 1
            if name == "stack28":
                print(f"oracle plan: stack28 {s.name} done", file=sys.stderr, flush=True)
        line = {"oracle_plan": name, "cores": cores, **host,
                "quantisers": {"oracle_s": round(stats["quant_s"], 2),
                               "oracle_GB_per_s": round(stats["quant_bytes"] / max(stats["quant_s"], 1e-9) / 1e9, 3),
                               "tensors": len(gpu_q), "parity": "bit-exact (codes and scales)"},
                "gemms_full": {"count": stats["gemms_full"], "oracle_s": round(stats["gemm_s_full"], 2),
                               "oracle_TFLOP_per_s": round(stats["gemm_flop_full"] / max(stats["gemm_s_full"], 1e-9)
                                                           / 1e12, 4)},
                "worst_rel_fro_vs_oracle": stats["worst_rel_fro"]}
        if stats["gemms_sampled"]:
            line["gemms_sampled_1_in_16_tiles"] = {
                "count": stats["gemms_sampled"], "oracle_s": round(stats["gemm_s_sampled"], 2),
                "oracle_TFLOP_per_s": round(stats["gemm_flop_sampled"] / max(stats["gemm_s_sampled"], 1e-9) / 1e12, 4),
                "oracle_s_for_all_tiles_extrapolated": round(stats["gemm_s_extrapolated"], 1)}
        print(json.dumps(line), flush=True)
        del cache
        torch.cuda.empty_cache()
    return 0


def per_kernel_protocol(args):
    """Each ABI call of one stack28 layer (the batched weight quantiser, then
    per linear the activation quantiser and FPROP; backward: the output
    gradient quantiser, DGRAD and WGRAD) timed alone: 10 warm-up calls, then
    50 timed calls, each preceded by a 256 MB write that evicts L2, with CUDA
    events on the launching stream around the call only.  Prints one JSON line
    with the median per call and its rate against the burst peaks (the kernels
    run alone, unthrottled) and, for the GEMMs, the rate scaled to the
    sustained peak's clock as well."""
    import torch
    from blockwise_fp8_linear_quantise_b300 import build as bld, ops, workloads
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    dev = torch.device("cuda", 0)
    bld.build()
    wl = workloads.make("stack28")
    specs = linear_list(wl, 1)
    runner = StackRunner(wl, specs, dev, args.scale_mode, False, False)
    runner.step()
    torch.cuda.synchronize()
    if ops.sync_status() != 0:
        raise SystemExit("device status not ok")
    peaks, basis = load_peaks()
    fp8_burst = peaks["bf16_tflops"] * FP8_PER_BF16
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(gpu_uuid(dev))
    clocks.start()
    rows = []
    for kind, work, fn, cargs in runner.calls:
        for _ in range(10):
            if fn(*cargs, stream.cuda_stream) != 0:
                raise SystemExit(f"{kind}: call failed")
        times = []
        for i in range(50):
            flush.fill_(i & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn(*cargs, stream.cuda_stream)
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) * 1e-3)
        t = statistics.median(times)
        gemm = kind in ("fprop", "dgrad", "wgrad")
        rate = work / t / (1e12 if gemm else 1e9)
        peak = fp8_burst if gemm else peaks["hbm_gbs"]
        rows.append({"call": kind, "work": work, "median_us": round(t * 1e6, 2),
                     ("TFLOP/s" if gemm else "GB/s"): round(rate, 1), "frac_of_burst": round(rate / peak, 4)})
    clk = clocks.stop()
    if ops.sync_status() != 0:
        raise SystemExit("device status not ok after the protocol")
    shapes = [[s.M, s.N, s.K] for s in specs]
    print(json.dumps({"per_kernel_protocol": "stack28 layer 0", "shapes_MNK": shapes, "scale_mode": args.scale_mode,
                      "protocol": "10 warm-up calls, median of 50, 256 MB L2 flush before each timed call",
                      "peaks": {"fp8_burst_TFLOP/s": round(fp8_burst, 1), "hbm_GB/s": peaks["hbm_gbs"],
                                "basis": f"{basis}: 2 x bf16 burst; HBM copy"},
                      "clocks": clk, "calls": rows}), flush=True)
    return 0


def mx_probe(args):
    """The MXFP8 1x32 recipe against the blockwise 1x128 / 128x128 recipe on
    the mlp_down layer (X [8192, 6144], W [2048, 6144], dY [8192, 2048]):
    for FPROP, DGRAD and WGRAD, the relative Frobenius error of each recipe's
    bf16 output against the unquantised bf16 operands' product (fp64 on the
    GPU, a measurement reference only), and the median time of each recipe's
    quantisers and GEMMs over 10 calls after 3 warm-up calls."""
    import torch
    from blockwise_fp8_linear_quantise_b300 import ops, workloads
    wl = workloads.make("mlp_down")
    X, W, dY = (workloads.tensor(wl, t).to("cuda") for t in ("x", "w", "dy"))
    M, K = X.shape
    N = W.shape[0]

    def med_ms(fn, n=10):
        for _ in range(3):
            fn()
        times = []
        for _ in range(n):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        return statistics.median(times)

    exact = {"fprop": X.double() @ W.double().t(), "dgrad": dY.double() @ W.double(),
             "wgrad": dY.double().t() @ X.double()}
    rel = lambda got, want: float(torch.linalg.norm(got.double() - want) / torch.linalg.norm(want))
    # blockwise recipe
    bq = {}
    q_block = lambda: (ops.quantize_act_1x128(X, rows=True, tokens=True), ops.quantize_w_128x128(W),
                       ops.quantize_act_1x128(dY, rows=True, tokens=True))
    (Xq, sX, XqT, sXT), (Wq, WqT, sW), (dYq, sdY, dYqT, sdYT) = q_block()
    bgemm = {"fprop": lambda: ops.fp8_block_gemm(ops.FPROP, Xq, sX, Wq, sW),
             "dgrad": lambda: ops.fp8_block_gemm(ops.DGRAD, dYq, sdY, WqT, sW),
             "wgrad": lambda: ops.fp8_block_gemm(ops.WGRAD, dYqT, sdYT, XqT, sXT)}
    # MXFP8 1x32 recipe
    q_mx = lambda: (ops.quantize_mx_1x32(X, rows=True, tokens=True), ops.quantize_mx_1x32(W, rows=True, tokens=True),
                    ops.quantize_mx_1x32(dY, rows=True, tokens=True))
    (mXq, msX, mXqT, msXT), (mWq, msW, mWqT, msWT), (mdYq, msdY, mdYqT, msdYT) = q_mx()
    mgemm = {"fprop": lambda: ops.mx_gemm(mXq, msX, mWq, msW), "dgrad": lambda: ops.mx_gemm(mdYq, msdY, mWqT, msWT),
             "wgrad": lambda: ops.mx_gemm(mdYqT, msdYT, mXqT, msXT)}
    out = {"probe": "mxfp8_1x32_vs_blockwise", "workload": f"mlp_down X [{M}, {K}], W [{N}, {K}], dY [{M}, {N}]",
           "quantise_ms": {"blockwise": round(med_ms(q_block), 4), "mx_1x32": round(med_ms(q_mx), 4)},
           "gemm": {}}
    for name in ("fprop", "dgrad", "wgrad"):
        Mg, Ng = exact[name].shape
        Kg = K if name == "fprop" else (N if name == "dgrad" else M)
        flop = 2.0 * Mg * Ng * Kg
        tb, tm = med_ms(bgemm[name]), med_ms(mgemm[name])
        out["gemm"][name] = {"rel_fro_err_vs_unquantised": {"blockwise": rel(bgemm[name](), exact[name]),
                                                             "mx_1x32": rel(mgemm[name](), exact[name])},
                             "TFLOP/s": {"blockwise": round(flop / (tb * 1e-3) / 1e12, 1),
                                         "mx_1x32": round(flop / (tm * 1e-3) / 1e12, 1)}}
    assert ops.sync_status() == 0
    print(json.dumps(out), flush=True)
    return 0


def swiglu_probe(args):
    """The SiLU-gated prologue on the down projection's input, gate+up output
    gu [8192, 12288] drawn as the mlp_down recipe (G, U ~ 0.5 t(4)): both
    1x128 quantisations of h [8192, 6144], no copy of h.  CUDA events over 20
    calls after 3 warm-up calls; the 201 MB input is larger than L2."""
    import torch
    from blockwise_fp8_linear_quantise_b300 import ops, workloads
    wl = workloads.make("mlp_down")
    gu = workloads.tensor(wl, "gu").to("cuda")
    M, F = gu.shape[0], gu.shape[1] // 2
    outs = ops.swiglu_quantize_1x128(gu, scale_mode=args.scale_mode)
    call = lambda: ops.swiglu_quantize_1x128(gu, h=None, q=outs[1], s=outs[2], qT=outs[3], sT=outs[4],
                                             scale_mode=args.scale_mode)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    assert ops.sync_status() == 0
    clocks = ClockSampler(gpu_uuid(gu.device))
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    n = 20
    e0.record()
    for _ in range(n):
        call()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert ops.sync_status() == 0
    us = e0.elapsed_time(e1) * 1e3 / n
    per_elem = 4 + 2 + 8 / 128  # g and u read, two codes and two scales per 128 written
    nbytes = M * F * per_elem
    peaks, basis = load_peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    line = {"probe": "swiglu_quantize_1x128", "workload": f"gu [{M}, {2 * F}] -> h [{M}, {F}], rows + tokens",
            "scale_mode": args.scale_mode, "us_per_call": round(us, 2), "bytes_per_call": int(nbytes),
            "value": round(gbs, 1), "unit": "GB/s", "peak": peaks["hbm_gbs"], "frac": round(gbs / peaks["hbm_gbs"], 4),
            "peak_basis": f"{basis} HBM copy", "clocks": clk,
            "unfused_bytes_per_call": int(M * F * (per_elem + 4)),
            "note": "unfused, h would be written and read back: 4 more bytes per element"}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.probe_fp8_peak:
        return fp8_peak_probe()
    if args.probe_swiglu:
        return swiglu_probe(args)
    if args.probe_mx:
        return mx_probe(args)
    if args.per_kernel:
        return per_kernel_protocol(args)
    if args.oracle_plan:
        return oracle_plan(args)
    if args.impl == "reference":
        return reference_arm(args)
    return gpu_arm(args)


if __name__ == "__main__":
    sys.exit(main())
