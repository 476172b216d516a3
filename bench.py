#!/usr/bin/env python
"""Benchmark of the NF4 double-quant QLoRA hot path on one Llama-3-8B-shaped layer.

One step = the whole hot path over the layer's 7 projections (q, k, v, o, gate,
up, down; 4096 tokens, rank 16, alpha 16, bf16 compute): for each projection
  nf4_quantize (bf16 master -> NF4 + double quant), nf4_dequantize (-> bf16),
  qlora_linear_fwd (T, y) and qlora_linear_bwd (G, dX, dA, dB),
all through the C ABI of libqlora_nf4.so.  value = fwd+bwd TFLOP/s over the whole
step (4MNK + 6Mr(N+K) per projection, no dW), so the quantize and dequantize time
counts against it.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 run under torchrun; each rank runs the same workload on its own GPU
(independent replicas, weak scaling, no data-path collective); a gloo barrier and
a max over ranks bracket the timed region.

--impl reference times the CPU oracle (oracle/) on the host cores on a bounded
sample of the same workload; rank 0 alone runs it.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD_NAME = "Llama-3-8B-shaped layer: q/o 4096x4096, k/v 1024x4096, gate/up 14336x4096, " \
                "down 4096x14336; NF4 double quant; QLoRA fwd+bwd on all 7, M=4096 (2x2048), r=16, alpha=16"
METRIC = "QLoRA NF4 linear fwd+bwd TFLOP/s and dequant weight GB/s vs roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--only", default=None,
                   help="restrict the step to one projection (for profiling; not a bench line)")
    p.add_argument("--cpu-sample-worker", type=float, default=None, help=argparse.SUPPRESS)
    p.add_argument("--profile-case", choices=("gate_linear", "small_m", "export", "smollm2"), default=None,
                   help="run one fixed workload for a profiler (no timing, no bench line): gate_linear = "
                        "quantize x2, dequantize x2, fwd x3, bwd x3 at the gate shape (M=4096, 14336x4096); "
                        "small_m = the 7-projection batched forward x4 at --tokens; export = embedding rows "
                        "and merged weight x2 each")
    p.add_argument("--tokens", type=int, default=1, help="M of --profile-case small_m")
    p.add_argument("--cpu-plan", action="store_true",
                   help="time the CPU oracle on workloads 1, 2, 4 and 5 with one thread and with every core "
                        "(one JSON line each); no GPU work")
    p.add_argument("--cpu-plan-max-log2", type=int, default=26,
                   help="largest 1-D size (log2) of workload 5 in --cpu-plan")
    p.add_argument("--cpu-plan-worker", default=None, help=argparse.SUPPRESS)
    p.add_argument("--traffic-json", default=None,
                   help="turn an ncu CSV (dram__bytes_read.sum, dram__bytes_write.sum, gpu__time_duration.sum "
                        "of the 14 bf16_tc_gemm launches of one bench step) into the per-launch traffic record")
    p.add_argument("--sweep", action="store_true",
                   help="time the other workloads (small-M forward, SmolLM2 stack, 1-D quantize and "
                        "dequantize sizes) and print one JSON line each; not the bench line")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---- distributed bookkeeping (host-side only) -------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo", rank=rank, world_size=world)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def gpu_local_cpus(dev):
    """The host CPUs that the kernel lists as local to this GPU's PCI function, or None.

    Pinned host pages land on the memory node of the thread that allocates them; on a
    machine with several host memory nodes, a node far from the GPU roughly halves the
    host-to-device copy rate, so the e2e buffers are allocated from a thread held here."""
    import torch
    p = torch.cuda.get_device_properties(dev)
    path = f"/sys/bus/pci/devices/{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0/local_cpulist"
    try:
        text = open(path).read().strip()
    except OSError:
        return None
    cpus = set()
    for part in text.split(","):
        if "-" in part:
            lo, hi = part.split("-")
            cpus.update(range(int(lo), int(hi) + 1))
        elif part:
            cpus.add(int(part))
    cpus &= os.sched_getaffinity(0)
    return cpus or None


# ---- clock sampling ---------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        rows = [r for t, r in self.rows if t0 <= t <= t1 and len(r) >= 9]
        if not rows:
            rows = [r for _, r in self.rows if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "", 1).isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ---- the workload -------------------------------------------------------------------

def linear_flops(M, N, K, r):
    """Algorithmic flops of one forward + backward: 4MNK (y and dX) + 6Mr(N+K) (T, s T B^T, G,
    s G A, dA, dB); the frozen base has no dW."""
    return 4 * M * N * K + 6 * M * r * (N + K)


def layer_flops(shapes, M, r):
    return sum(linear_flops(M, N, K, r) for _, N, K in shapes)


class Layer:
    """Device buffers for one step over the 7 projections (allocated once)."""

    def __init__(self, dev, seed_base=0, only=None):
        import torch
        from bit_nf4_quantized_gb300 import binding
        from bit_nf4_quantized_gb300 import workloads as wl
        c = wl.W3
        self.M, self.r, self.alpha = c["M"], c["r"], c["alpha"]
        self.shapes = [t for t in c["shapes"] if only is None or t[0] == only]
        if not self.shapes:
            raise ValueError(f"no projection named {only}")
        self.dev = dev
        self.proj = []
        lib = binding.load()
        max_w = max(N * K for _, N, K in self.shapes)
        self.deq = torch.empty(max_w, dtype=torch.bfloat16, device=dev)
        ws_q = max(lib.nf4_quantize_workspace_bytes(N * K, 1) for _, N, K in self.shapes)
        # the step decodes each weight once (the dequantize row) and both contractions read that
        # bf16 copy; decode_once = False runs the NF4-input calls, which decode once per call
        self.decode_once = True
        # decode_batch = True (the headline step) decodes all 7 weights in one
        # nf4_dequantize_batch call after the quantize (7 bf16 copies); False decodes each right
        # before its projection's calls
        self.decode_batch = True
        self.deq_all = None
        ws_f = max(lib.qlora_fwd_workspace_bytes(self.M, N, K, self.r, 1) for _, N, K in self.shapes)
        ws_b = max(lib.qlora_bwd_workspace_bytes(self.M, N, K, self.r, 1) for _, N, K in self.shapes)
        self.ws_q = torch.empty(max(ws_q, 16), dtype=torch.uint8, device=dev)
        self.ws_f = torch.empty(max(ws_f, 16), dtype=torch.uint8, device=dev)
        self.ws_b = torch.empty(max(ws_b, 16), dtype=torch.uint8, device=dev)
        # projections that read the same activation (q, k, v; gate, up) share one x tensor
        shared_x = {}
        for i, (name, N, K) in enumerate(self.shapes):
            seed = wl.seed_for(3, 100 * i) + seed_base
            p = dict(name=name, N=N, K=K, x_of=wl.LAYER_INPUTS.get(name, name))
            p["w"] = wl.device_student_t((N, K), c["t_df"], c["w_scale"], seed, dev, torch.bfloat16)
            if p["x_of"] not in shared_x:
                shared_x[p["x_of"]] = wl.device_normal((self.M, K), 1.0, seed + 1, dev, torch.bfloat16)
            p["x"] = shared_x[p["x_of"]]
            p["dy"] = wl.device_normal((self.M, N), 1.0, seed + 2, dev, torch.bfloat16)
            p["A"] = wl.device_normal((self.r, K), 1.0 / self.r, seed + 3, dev, torch.float32)
            p["B"] = wl.device_normal((N, self.r), 0.01, seed + 4, dev, torch.float32)
            p["q"] = binding.Nf4Tensor.empty((N, K), True, dev)
            p["y"] = torch.empty((self.M, N), dtype=torch.bfloat16, device=dev)
            p["T"] = torch.empty((self.M, self.r), dtype=torch.float32, device=dev)
            p["dx"] = torch.empty((self.M, K), dtype=torch.bfloat16, device=dev)
            p["dA"] = torch.empty((self.r, K), dtype=torch.float32, device=dev)
            p["dB"] = torch.empty((N, self.r), dtype=torch.float32, device=dev)
            self.proj.append(p)
        self.ws_qb = torch.empty(max(16, binding.nf4_quantize_batch_workspace_bytes(self.quant_pairs())),
                                 dtype=torch.uint8, device=dev)
        # the grouped calls (the headline step): one forward and one backward batch over the 7
        # projections with their weights decoded; consecutive projections with one x share a pass
        shapes = [(p["N"], p["K"]) for p in self.proj]
        xs = [p["x_of"] for p in self.proj]
        self.grouped = True
        self.ws_fb = torch.empty(max(16, binding.qlora_fwd_batch_workspace_bytes(self.M, shapes, self.r, xs=xs,
                                                                                 w16=True)),
                                 dtype=torch.uint8, device=dev)
        self.ws_bb = torch.empty(max(16, binding.qlora_bwd_batch_workspace_bytes(self.M, shapes, self.r, xs=xs,
                                                                                 w16=True)),
                                 dtype=torch.uint8, device=dev)
        # the activations once each (the e2e copies)
        self.x_first = {}
        for i, p in enumerate(self.proj):
            self.x_first.setdefault(p["x_of"], i)

    def quant_pairs(self):
        return [(p["w"], p["q"]) for p in self.proj]

    def quantize_all(self):
        """The layer's weights in one nf4_quantize_batch call."""
        from bit_nf4_quantized_gb300 import binding as b
        b.nf4_quantize_batch(self.quant_pairs(), workspace=self.ws_qb)

    def step_one(self, p, quantize=True):
        from bit_nf4_quantized_gb300 import binding as b
        if quantize:
            b.nf4_quantize(p["w"], True, out=p["q"], workspace=self.ws_q)
        w16 = self.deq[:p["N"] * p["K"]].view(p["N"], p["K"])
        b.nf4_dequantize(p["q"], out=w16)
        if self.decode_once:
            b.qlora_linear_fwd_w16(p["x"], w16, p["A"], p["B"], self.alpha, y=p["y"], T=p["T"],
                                   workspace=self.ws_f)
            b.qlora_linear_bwd_w16(p["dy"], p["x"], p["T"], w16, p["A"], p["B"], self.alpha, dx=p["dx"],
                                   dA=p["dA"], dB=p["dB"], workspace=self.ws_b)
            return
        b.qlora_linear_fwd(p["x"], p["q"], p["A"], p["B"], self.alpha, y=p["y"], T=p["T"],
                           workspace=self.ws_f)
        b.qlora_linear_bwd(p["dy"], p["x"], p["T"], p["q"], p["A"], p["B"], self.alpha, dx=p["dx"],
                           dA=p["dA"], dB=p["dB"], workspace=self.ws_b)

    def run_group(self, idx, quantize=True):
        """Projections idx (the whole layer, or one set that reads one x): quantize (one batch
        call), dequantize (one batch call), then one grouped forward and one grouped backward
        call reading the decoded weights."""
        import torch
        from bit_nf4_quantized_gb300 import binding as b
        if self.deq_all is None:
            self.deq_all = [torch.empty((p["N"], p["K"]), dtype=torch.bfloat16, device=self.dev) for p in self.proj]
        ps = [self.proj[i] for i in idx]
        if quantize:
            b.nf4_quantize_batch([(p["w"], p["q"]) for p in ps], workspace=self.ws_qb)
        b.nf4_dequantize_batch([(self.proj[i]["q"], self.deq_all[i]) for i in idx])
        b.qlora_linear_fwd_batch([dict(x=p["x"], w16=self.deq_all[i], A=p["A"], B=p["B"], alpha=self.alpha,
                                       y=p["y"], T=p["T"]) for i, p in zip(idx, ps)], workspace=self.ws_fb)
        b.qlora_linear_bwd_batch([dict(dy=p["dy"], x=p["x"], T=p["T"], w16=self.deq_all[i], A=p["A"], B=p["B"],
                                       alpha=self.alpha, dx=p["dx"], dA=p["dA"], dB=p["dB"])
                                  for i, p in zip(idx, ps)], workspace=self.ws_bb)

    def step(self):
        """One step: the layer's 7 weights quantized in one batch call and dequantized in one batch
        call, then one grouped forward and one grouped backward call (q, k, v and gate, up each
        share one pass over their x).  Variants: grouped = False runs per projection single
        forward and backward calls on the decoded weights; decode_batch = False decodes each
        weight right before its projection's single calls."""
        import torch
        from bit_nf4_quantized_gb300 import binding as b
        if self.grouped and self.decode_batch:
            self.run_group(list(range(len(self.proj))))
            return
        self.quantize_all()
        if not self.decode_batch:
            for p in self.proj:
                self.step_one(p, quantize=False)
            return
        if self.deq_all is None:
            self.deq_all = [torch.empty((p["N"], p["K"]), dtype=torch.bfloat16, device=self.dev) for p in self.proj]
        b.nf4_dequantize_batch([(p["q"], w16) for p, w16 in zip(self.proj, self.deq_all)])
        for p, w16 in zip(self.proj, self.deq_all):
            b.qlora_linear_fwd_w16(p["x"], w16, p["A"], p["B"], self.alpha, y=p["y"], T=p["T"],
                                   workspace=self.ws_f)
            b.qlora_linear_bwd_w16(p["dy"], p["x"], p["T"], w16, p["A"], p["B"], self.alpha, dx=p["dx"],
                                   dA=p["dA"], dB=p["dB"], workspace=self.ws_b)

    def x_groups(self):
        """Projection indices in runs that read one x (in order)."""
        out = []
        for i, p in enumerate(self.proj):
            if out and self.proj[out[-1][0]]["x_of"] == p["x_of"]:
                out[-1].append(i)
            else:
                out.append([i])
        return out

    @staticmethod
    def inputs_of(p):
        return [p[k] for k in ("w", "x", "dy")]

    @staticmethod
    def results_of(p):
        return [p[k] for k in ("dA", "dB")]

    def input_tensors(self):
        # a shared x once
        out = []
        for i, p in enumerate(self.proj):
            out += [p["w"], p["dy"]] + ([p["x"]] if self.x_first[p["x_of"]] == i else [])
        return out

    def result_tensors(self):
        return [t for p in self.proj for t in self.results_of(p)]


def gemm_traffic(kind):
    """DRAM bytes per launch of one GEMM kind, from the committed ncu capture of one bench
    step (profiles/bf16_tc_gemm_llama8b_step_traffic.json), or None once the kernel source
    differs from the one the counters were taken on."""
    import hashlib
    root = os.path.dirname(os.path.abspath(__file__))
    try:
        with open(os.path.join(root, "profiles", "bf16_tc_gemm_llama8b_step_traffic.json")) as f:
            rec = json.load(f)
        with open(os.path.join(root, "bit_nf4_quantized_gb300", "csrc", "linear_tc.cu"), "rb") as f:
            src = hashlib.sha256(f.read()).hexdigest()
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != src:
        return None
    return rec.get("per_launch_bytes", {}).get(kind)


def clock_normalised(achieved, clocks, peak_sus, pk):
    """TFLOP/s per MHz of the median SM clock of the bench's timed region, against the same
    for the sustained peak run and the median SM clock it recorded."""
    mhz = clocks.get("sm_mhz")
    peak_mhz = (pk.get("clocks_under_load") or {}).get("sm_mhz_median")
    if not mhz or not peak_mhz or not peak_sus:
        return None
    return {"kernel_sm_mhz": mhz, "peak_run_sm_mhz": peak_mhz,
            "achieved_per_mhz": achieved / mhz, "sustained_peak_per_mhz": peak_sus / peak_mhz,
            "frac": (achieved / mhz) / (peak_sus / peak_mhz)}


def time_steps(fn, steps, stream):
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end)


# ---- CPU oracle sample (cpu_baseline and the reference arm) --------------------------

def oracle_sample():
    """One bounded sample of the same step on the CPU oracle: the k_proj weight rows
    0..255 (256 x 4096 slice) quantized, dequantized, and QLoRA fwd+bwd for 512 tokens."""
    import numpy as np
    from bit_nf4_quantized_gb300 import workloads as wl
    from oracle import nf4 as onf4
    from oracle import qlora
    c = wl.W3
    N, K, M, r = 256, 4096, 512, c["r"]
    w = wl.student_t((N, K), c["t_df"], c["w_scale"], 3, 777)
    x = wl.normal((M, K), 1.0, 3, 778)
    dy = wl.normal((M, N), 1.0, 3, 779)
    A, B = wl.adapters(N, K, r, 3, 780)
    s = qlora.lora_scale(c["alpha"], r)

    def run():
        q = onf4.quantize(w, double_quant=True)
        wd = onf4.dequantize(q, "f32").reshape(N, K)
        _ = onf4.dequantize(q, "bf16")
        qlora.forward(x, wd, A, B, s, "bf16")
        qlora.backward(dy, x, wd, A, B, s, "bf16")
    return run, linear_flops(M, N, K, r), "k_proj rows 0..255 (256x4096 slice): quantize, dequantize " \
        "(f32 and bf16), fwd+bwd at M=512, r=16; float64 numpy oracle"


def _thread_env(threads):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = str(threads)
    return env


def cpu_sample_worker(budget_s):
    """Child process: time the oracle sample for about budget_s seconds, print JSON."""
    run, flops, sample = oracle_sample()
    run()   # warm
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < budget_s or n == 0:
        run()
        n += 1
    dt = (time.perf_counter() - t0) / n
    print(json.dumps({"seconds_per_sample": dt, "repetitions": n, "flops": flops, "sample": sample}))
    return 0


def time_oracle_sample(threads, budget_s):
    """The oracle sample in a child process whose BLAS is limited to `threads` threads."""
    out = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample-worker", str(budget_s)],
                         env=_thread_env(threads), capture_output=True, text=True, check=True)
    return json.loads(out.stdout.strip().splitlines()[-1])


def cpu_baseline(budget_s=12.0):
    """The oracle as it stands on this host's cores: one bounded sample of the step, timed with
    all cores and with one thread (each about budget_s / 2 seconds), and the time one whole
    config-3 step would take at those rates (the oracle's cost is its float64 products, which
    scale with the flops)."""
    cores = os.cpu_count() or 1
    allc = time_oracle_sample(cores, budget_s / 2)
    one = time_oracle_sample(1, budget_s / 2)
    from bit_nf4_quantized_gb300 import workloads as wl
    c = wl.W3
    step = layer_flops(c["shapes"], c["M"], c["r"])
    rate_all = allc["flops"] / allc["seconds_per_sample"]
    rate_one = one["flops"] / one["seconds_per_sample"]
    return {"value": rate_all / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{allc['sample']}; {allc['repetitions']} repetitions, "
                      f"{allc['seconds_per_sample']:.3f} s each",
            "single_thread": {"value": rate_one / 1e12, "unit": "TFLOP/s", "cores": 1,
                              "seconds_per_sample": one["seconds_per_sample"]},
            "extrapolated_step_s": {"all_cores": step / rate_all, "single_thread": step / rate_one,
                                    "of": "one Llama-3-8B-shaped layer step (7 projections, M=4096), "
                                          "extrapolated by flops from the sample"}}


def cpu_plan_worker(which, max_log2):
    """Child process: one workload of --cpu-plan on the oracle, timed; prints JSON lines."""
    import numpy as np
    from bit_nf4_quantized_gb300 import workloads as wl
    from oracle import nf4 as onf4
    from oracle import qlora

    def timed(fn):
        t0 = time.perf_counter()
        out = fn()
        return time.perf_counter() - t0, out

    def emit(d):
        print(json.dumps(d), flush=True)

    if which == "1":
        c = wl.W1
        N, K, M, r = c["N"], c["K"], c["M"], c["r"]
        w = wl.normal((N, K), c["w_std"], 1, 0)
        x, dy = wl.normal((M, K), 1.0, 1, 1), wl.normal((M, N), 1.0, 1, 2)
        A, B = wl.adapters(N, K, r, 1, 3)
        s = qlora.lora_scale(c["alpha"], r)

        def run():
            q = onf4.quantize(w, double_quant=True)
            wd = onf4.dequantize(q, "f32").reshape(N, K)
            qlora.forward(x, wd, A, B, s, "f32")
            qlora.backward(dy, x, wd, A, B, s, "f32")
        run()
        dt, _ = timed(run)
        emit({"workload": c["name"], "seconds": dt, "GFLOP/s": linear_flops(M, N, K, r) / dt / 1e9,
              "covers": "quantize + dequantize + fwd + bwd (fp32 operands, float64 products)"})
    elif which == "2":
        c = wl.W2
        M, r = c["M"], c["r"]
        s = qlora.lora_scale(c["alpha"], r)
        mats = []
        for j, (name, N, K) in enumerate(c["shapes"]):
            if name in c["targets"]:
                q = onf4.quantize(wl.normal((N, K), c["w_std"], 2, 2000 + j), double_quant=True)
                A, B = wl.adapters(N, K, r, 2, 2100 + j)
                mats.append((N, K, q, A, B, wl.normal((M, K), 1.0, 2, 2200 + j), wl.normal((M, N), 1.0, 2, 2300 + j)))

        def layer():
            for N, K, q, A, B, x, dy in mats:
                wd = onf4.dequantize(q, "f32").reshape(N, K)
                qlora.forward(x, wd, A, B, s, "bf16")
                qlora.backward(dy, x, wd, A, B, s, "bf16")
        layer()
        dt, _ = timed(layer)
        flops = sum(linear_flops(M, N, K, r) for N, K, *_ in mats)
        emit({"workload": c["name"], "seconds_per_step": dt * c["layers"], "GFLOP/s": flops / dt / 1e9,
              "covers": "per layer: dequantize + fwd + bwd of q and v; one layer timed, x 30 layers"})
    elif which == "4":
        c = wl.W4
        r = c["r"]
        s = qlora.lora_scale(c["alpha"], r)
        dec_s = 0.0
        decoded = []
        for i, (_, N, K) in enumerate(c["shapes"]):
            n = N * K
            parts = wl.random_nf4_parts((n + 1) // 2, onf4.num_blocks(n), onf4.num_nested(n), True, 4, 700 + i)
            ref = dict(numel=n, double_quant=True, packed=parts["packed"], absmax=parts["absmax"],
                       nested=parts["nested"], offset=parts["offset"])
            dt, wd = timed(lambda: onf4.dequantize(ref, "f32").reshape(N, K))
            dec_s += dt
            A, B = wl.adapters(N, K, r, 4, 710 + i)
            decoded.append((N, K, wd, A, B))
        wbytes = sum(onf4.packed_bytes(N * K, True) for N, K, *_ in decoded)
        for M in c["Ms"]:
            def fwd():
                for N, K, wd, A, B in decoded:
                    qlora.forward(wl.normal((M, K), 1.0, 4, 720 + M), wd, A, B, s, "bf16")
            dt, _ = timed(fwd)
            emit({"workload": c["name"], "tokens": M, "seconds_per_layer": dec_s + dt,
                  "weight_GB/s": wbytes / (dec_s + dt) / 1e9, "dequantize_seconds": dec_s,
                  "covers": "dequantize of the 7 stored weights + forward (the oracle needs the decoded weight)"})
    elif which == "5":
        c = wl.W5
        for n in [v for v in c["sizes"] if v <= (1 << max_log2)]:
            x = wl.with_outliers(wl.normal(n, c["std"], 5, 1), c["outlier_frac"], c["outlier_mult"], 5, 2)
            tq, q = timed(lambda: onf4.quantize(x, double_quant=True))
            td, _ = timed(lambda: onf4.dequantize(q, "f32"))
            stored = onf4.packed_bytes(n, True)
            emit({"workload": c["name"], "numel": n, "quantize_GB/s": (4 * n + stored + 4) / tq / 1e9,
                  "dequantize_GB/s": (stored + 4 * n) / td / 1e9, "quantize_s": tq, "dequantize_s": td})
    return 0


def cpu_plan(args):
    """The oracle on workloads 1, 2, 4 and 5, each in a child process with one BLAS thread and
    with every core (core count of this host stated); workload 3 is the bench line's sample."""
    cores = os.cpu_count() or 1
    for which in ("1", "2", "4", "5"):
        for threads in (1, cores):
            out = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-plan-worker", which,
                                  "--cpu-plan-max-log2", str(args.cpu_plan_max_log2)],
                                 env=_thread_env(threads), capture_output=True, text=True, check=True)
            for line in out.stdout.strip().splitlines():
                d = json.loads(line)
                d.update({"cpu_plan": "oracle", "threads": threads, "host_cores": cores})
                print(json.dumps(d), flush=True)
    return 0


def reference_arm(args, rank, world):
    if rank != 0:
        return 0
    run, flops, sample = oracle_sample()
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    total = time.perf_counter() - t0
    v = flops * args.steps / total / 1e12
    cores = os.cpu_count() or 1
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD_NAME, "reference_sample": sample},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---- main ---------------------------------------------------------------------------

def random_stored_nf4(shape, seed, dev):
    """An NF4 tensor of random stored bytes on the device (codes, scale codes, nested
    maxima in U(0.01, 0.05), offset 0.03): any byte pattern is a valid stored tensor."""
    import torch
    from bit_nf4_quantized_gb300 import binding as bq
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    q = bq.Nf4Tensor.empty(shape, True, dev)
    q.packed.copy_(torch.randint(0, 256, q.packed.shape, generator=g, device=dev, dtype=torch.uint8))
    q.absmax.copy_(torch.randint(0, 256, q.absmax.shape, generator=g, device=dev, dtype=torch.uint8))
    q.nested_absmax.copy_(torch.rand(q.nested_absmax.shape, generator=g, device=dev) * 0.04 + 0.01)
    q.offset[0] = 0.03
    return q


def measure_no_double_quant(layer, row_ms):
    """The gate projection's forward + backward with its double-quantized weight and with a
    copy holding fp32 block maxima instead (same kernels, the plain scale); each timed as a
    graph with L2 flushed between replays."""
    from bit_nf4_quantized_gb300 import binding as bq
    p = next(q for q in layer.proj if q["name"] == "gate_proj")
    q_plain = bq.nf4_quantize(p["w"], double_quant=False)

    def fwd_bwd(q):
        bq.qlora_linear_fwd(p["x"], q, p["A"], p["B"], layer.alpha, y=p["y"], T=p["T"], workspace=layer.ws_f)
        bq.qlora_linear_bwd(p["dy"], p["x"], p["T"], q, p["A"], p["B"], layer.alpha, dx=p["dx"], dA=p["dA"],
                            dB=p["dB"], workspace=layer.ws_b)

    flops = layer_flops([("gate_proj", p["N"], p["K"])], layer.M, layer.r)
    ms_dq = row_ms(lambda: fwd_bwd(p["q"]))
    ms_plain = row_ms(lambda: fwd_bwd(q_plain))
    return {"shape": [p["N"], p["K"]], "tokens": layer.M,
            "TFLOP/s_double_quant": flops / (ms_dq / 1e3) / 1e12,
            "TFLOP/s_fp32_absmax": flops / (ms_plain / 1e3) / 1e12,
            "ms_double_quant": ms_dq, "ms_fp32_absmax": ms_plain,
            "timing": "fwd+bwd of one projection as a graph, L2 flushed between replays"}


def measure_f16_profile(layer, row_ms):
    """The gate projection's forward + backward in the FP16 compute profile (IEEE half operands
    and outputs, fp32 accumulation) beside the bf16 one, same weight, each as a graph with L2
    flushed between replays."""
    import torch
    from bit_nf4_quantized_gb300 import binding as bq
    p = next(q for q in layer.proj if q["name"] == "gate_proj")
    x16, dy16 = p["x"].to(torch.float16), p["dy"].to(torch.float16)
    y16, dx16 = torch.empty_like(p["y"], dtype=torch.float16), torch.empty_like(p["dx"], dtype=torch.float16)

    def fwd_bwd(x, dy, y, dx):
        bq.qlora_linear_fwd(x, p["q"], p["A"], p["B"], layer.alpha, y=y, T=p["T"], workspace=layer.ws_f)
        bq.qlora_linear_bwd(dy, x, p["T"], p["q"], p["A"], p["B"], layer.alpha, dx=dx, dA=p["dA"], dB=p["dB"],
                            workspace=layer.ws_b)

    flops = layer_flops([("gate_proj", p["N"], p["K"])], layer.M, layer.r)
    ms16 = row_ms(lambda: fwd_bwd(x16, dy16, y16, dx16))
    msb = row_ms(lambda: fwd_bwd(p["x"], p["dy"], p["y"], p["dx"]))
    return {"shape": [p["N"], p["K"]], "tokens": layer.M, "TFLOP/s_f16": flops / (ms16 / 1e3) / 1e12,
            "TFLOP/s_bf16": flops / (msb / 1e3) / 1e12, "ms_f16": ms16, "ms_bf16": msb,
            "timing": "fwd+bwd of one projection as a graph, L2 flushed between replays"}


def measure_export_rows(dev, row_ms, hbm):
    """The selected-row embedding decode and the merged-weight export, each one call timed
    as a replayed graph with L2 flushed between replays; GB/s of algorithmic bytes."""
    import torch
    from bit_nf4_quantized_gb300 import binding as bq
    from bit_nf4_quantized_gb300 import workloads as wl
    lib = bq.load()
    e = wl.W6
    rows, dim, n_ids = e["rows"], e["dim"], e["n_ids"]
    table = random_stored_nf4((rows, dim), wl.seed_for(6, 10), dev)
    g = torch.Generator(device=dev)
    g.manual_seed(wl.seed_for(6, 11))
    ids = torch.randint(0, rows, (n_ids,), generator=g, device=dev, dtype=torch.int64)
    rows_out = torch.empty((n_ids, dim), dtype=torch.bfloat16, device=dev)
    # per id: dim/2 code bytes, dim/64 scale codes, one 4-byte nested maximum (a 4096-wide
    # row lies in one 16384-element group), the 8-byte id and dim bf16 outputs
    emb_bytes = n_ids * (dim // 2 + dim // 64 + 4 + 8 + 2 * dim)
    emb_ms = row_ms(lambda: bq.nf4_embedding_rows(table, ids, out=rows_out), reps=20)
    # the store floor: filling the same output buffer (a library fill kernel), timed the same
    # way; after the flush L2 holds dirty lines, so every output line written evicts one
    emb_floor_ms = row_ms(lambda: rows_out.zero_(), reps=20)
    del table, rows_out

    m = wl.W7
    N, K, r = m["N"], m["K"], m["r"]
    W = random_stored_nf4((N, K), wl.seed_for(7, 20), dev)
    A = wl.device_normal((r, K), 1.0 / r, wl.seed_for(7, 21), dev, torch.float32)
    B = wl.device_normal((N, r), 0.01, wl.seed_for(7, 22), dev, torch.float32)
    merged = torch.empty((N, K), dtype=torch.float32, device=dev)
    merge_bytes = lib.nf4_packed_bytes(N * K, 1) + 4 * r * K + 4 * N * r + 4 * N * K
    merge_ms = row_ms(lambda: bq.nf4_merge_lora(W, A, B, m["alpha"], out=merged), reps=20)
    merge_floor_ms = row_ms(lambda: merged.zero_(), reps=20)
    del W, merged
    emb_gbs = emb_bytes / (emb_ms / 1e3) / 1e9
    merge_gbs = merge_bytes / (merge_ms / 1e3) / 1e9
    return {
        "embedding": {"GB/s": emb_gbs, "frac": emb_gbs / hbm, "bytes_per_call": emb_bytes, "ms_per_call": emb_ms,
                      "store_floor_ms": emb_floor_ms, "frac_of_store_floor": emb_floor_ms / emb_ms,
                      "workload": e["name"], "timing": "one call as a graph, L2 flushed between replays"},
        "merge": {"GB/s": merge_gbs, "frac": merge_gbs / hbm, "bytes_per_call": merge_bytes,
                  "ms_per_call": merge_ms, "store_floor_ms": merge_floor_ms,
                  "frac_of_store_floor": merge_floor_ms / merge_ms, "workload": m["name"],
                  "timing": "one call as a graph, L2 flushed between replays; store_floor_ms = zero-filling "
                            "the same output the same way"},
    }


def measure_small_m(layer, row_ms, hbm):
    """The decode-like small-M forward on the same 7 quantized matrices (r = 8, alpha = 16):
    the whole layer through one qlora_linear_fwd_batch call, per M, as a replayed graph with L2
    flushed; GB/s over the stored weight bytes the call must read."""
    import torch
    from bit_nf4_quantized_gb300 import binding as bq
    from bit_nf4_quantized_gb300 import workloads as wl
    c = wl.W4
    r, alpha, Ms = c["r"], c["alpha"], c["Ms"]
    dev = layer.dev
    lib = bq.load()
    mmax = max(Ms)
    shapes = [(p["N"], p["K"]) for p in layer.proj]
    ws = torch.empty(max(16, max(bq.qlora_fwd_batch_workspace_bytes(m, shapes, r) for m in Ms)), dtype=torch.uint8,
                     device=dev)
    ad = []
    for i, p in enumerate(layer.proj):
        seed = wl.seed_for(4, 100 * i)
        ad.append(dict(x=wl.device_normal((mmax, p["K"]), 1.0, seed + 1, dev, torch.bfloat16),
                       A=wl.device_normal((r, p["K"]), 1.0 / r, seed + 3, dev, torch.float32),
                       B=wl.device_normal((p["N"], r), 0.01, seed + 4, dev, torch.float32),
                       y=torch.empty((mmax, p["N"]), dtype=torch.bfloat16, device=dev),
                       T=torch.empty((mmax, r), dtype=torch.float32, device=dev)))
    wbytes = sum(lib.nf4_packed_bytes(p["N"] * p["K"], 1) for p in layer.proj)
    out = {}
    for m in Ms:
        items = [dict(x=a["x"][:m], W=p["q"], A=a["A"], B=a["B"], alpha=alpha, y=a["y"][:m], T=a["T"][:m])
                 for p, a in zip(layer.proj, ad)]
        ms = row_ms(lambda: bq.qlora_linear_fwd_batch(items, workspace=ws), reps=20)
        gbs = wbytes / (ms / 1e3) / 1e9
        out[str(m)] = {"us_per_layer": ms * 1e3, "weight_GB/s": gbs, "frac": gbs / hbm}
    return {"per_M": out, "weight_bytes_per_layer": wbytes, "peak_gbs": hbm,
            "workload": c["name"] + ", the 7 projections in one qlora_linear_fwd_batch call",
            "timing": "one call as a graph, L2 flushed between replays"}


def measure_fp32_576(dev, row_ms):
    """Workload 1: one 576 x 576 weight, fp32 profile, QLoRA fwd+bwd at M = 512, r = 16,
    alpha = 32; microseconds per fwd+bwd (a graph of the two calls, L2 flushed)."""
    import torch
    from bit_nf4_quantized_gb300 import binding as bq
    from bit_nf4_quantized_gb300 import workloads as wl
    c = wl.W1
    N, K, M, r = c["N"], c["K"], c["M"], c["r"]
    q = bq.nf4_quantize(wl.device_normal((N, K), c["w_std"], wl.seed_for(1, 0), dev, torch.float32), True)
    x = wl.device_normal((M, K), 1.0, wl.seed_for(1, 1), dev, torch.float32)
    dy = wl.device_normal((M, N), 1.0, wl.seed_for(1, 2), dev, torch.float32)
    A = wl.device_normal((r, K), 1.0 / r, wl.seed_for(1, 3), dev, torch.float32)
    B = wl.device_normal((N, r), 0.01, wl.seed_for(1, 4), dev, torch.float32)
    y, T = bq.qlora_linear_fwd(x, q, A, B, c["alpha"])
    dx, dA, dB = bq.qlora_linear_bwd(dy, x, T, q, A, B, c["alpha"])

    def fwd_bwd():
        bq.qlora_linear_fwd(x, q, A, B, c["alpha"], y=y, T=T)
        bq.qlora_linear_bwd(dy, x, T, q, A, B, c["alpha"], dx=dx, dA=dA, dB=dB)
    ms = row_ms(fwd_bwd, reps=20)
    flops = linear_flops(M, N, K, r)
    return {"us_per_fwd_bwd": ms * 1e3, "TFLOP/s": flops / (ms / 1e3) / 1e12, "flops": flops,
            "workload": c["name"], "timing": "fwd+bwd as one graph, L2 flushed between replays",
            "context": "pages: 0.1346 ms for the fused FP32 576x576 linear at 32 tokens on a Tesla V100 "
                       "(V100 accelerated qualification record, component_benchmarks[0])"}


def graph_ms(fn, dev, stream, flush, reps=10):
    """Median milliseconds of `fn` captured as one CUDA graph and replayed, with L2 flushed
    (a 256 MB write) before every replay, outside the timed interval."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    torch.cuda.synchronize(dev)
    ts = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    ts.sort()
    return ts[len(ts) // 2]


def measure_smollm2(dev, time_ms, tc):
    """The SmolLM2-135M-shaped stack (workload 2): forward + backward of q and v in each of 30
    layers at M = 512, r = 16, bf16.  Within a layer q and v read the same x.  Timed two ways,
    each as one graph: per layer one qlora_linear_fwd_batch and one qlora_linear_bwd_batch over
    (q, v) (the grouped launches), and one qlora_linear_fwd + qlora_linear_bwd call per
    projection."""
    import torch
    from bit_nf4_quantized_gb300 import binding as bq
    from bit_nf4_quantized_gb300 import workloads as wl
    lib = bq.load()
    c = wl.W2
    M, r, alpha = c["M"], c["r"], c["alpha"]
    targets = [(n, N, K) for n, N, K in c["shapes"] if n in c["targets"]]
    shapes = [(N, K) for _, N, K in targets]
    ws = torch.empty(max(16, max(lib.qlora_fwd_workspace_bytes(M, N, K, r, 1) for N, K in shapes),
                         max(lib.qlora_bwd_workspace_bytes(M, N, K, r, 1) for N, K in shapes),
                         bq.qlora_bwd_batch_workspace_bytes(M, shapes, r),
                         bq.qlora_fwd_batch_workspace_bytes(M, shapes, r)), dtype=torch.uint8, device=dev)
    K0 = targets[0][2]
    x = wl.device_normal((M, K0), 1.0, wl.seed_for(2, 1), dev, torch.bfloat16)   # the layer input, shared
    bufs = []
    for j, (_, N, K) in enumerate(targets):
        seed = wl.seed_for(2, 10 * j)
        bufs.append(dict(dy=wl.device_normal((M, N), 1.0, seed + 2, dev, torch.bfloat16),
                         y=torch.empty((M, N), dtype=torch.bfloat16, device=dev),
                         T=torch.empty((M, r), dtype=torch.float32, device=dev),
                         dx=torch.empty((M, K), dtype=torch.bfloat16, device=dev),
                         dA=torch.empty((r, K), dtype=torch.float32, device=dev),
                         dB=torch.empty((N, r), dtype=torch.float32, device=dev)))
    layers = []
    for layer in range(c["layers"]):
        mats = []
        for j, (_, N, K) in enumerate(targets):
            seed = wl.seed_for(2, 1000 + 10 * (layer * len(targets) + j))
            mats.append(dict(q=bq.nf4_quantize(wl.device_normal((N, K), 0.02, seed, dev, torch.bfloat16), True),
                             A=wl.device_normal((r, K), 1.0 / r, seed + 3, dev, torch.float32),
                             B=wl.device_normal((N, r), 0.01, seed + 4, dev, torch.float32)))
        layers.append(mats)

    def grouped():
        for mats in layers:
            bq.qlora_linear_fwd_batch([dict(x=x, W=m["q"], A=m["A"], B=m["B"], alpha=alpha, y=b["y"], T=b["T"])
                                       for m, b in zip(mats, bufs)], workspace=ws)
            bq.qlora_linear_bwd_batch([dict(dy=b["dy"], x=x, T=b["T"], W=m["q"], A=m["A"], B=m["B"], alpha=alpha,
                                            dx=b["dx"], dA=b["dA"], dB=b["dB"]) for m, b in zip(mats, bufs)],
                                      workspace=ws)

    def single():
        for mats in layers:
            for m, b in zip(mats, bufs):
                bq.qlora_linear_fwd(x, m["q"], m["A"], m["B"], alpha, y=b["y"], T=b["T"], workspace=ws)
                bq.qlora_linear_bwd(b["dy"], x, b["T"], m["q"], m["A"], m["B"], alpha, dx=b["dx"], dA=b["dA"],
                                    dB=b["dB"], workspace=ws)

    launches0 = bq.launch_count()
    grouped()
    torch.cuda.synchronize(dev)
    launches = bq.launch_count() - launches0
    ms_g = time_ms(grouped)
    ms_s = time_ms(single)
    flops = sum(linear_flops(M, N, K, r) for mats in layers for (N, K) in shapes)
    if bq.device_status() != bq.NF4_OK:
        raise RuntimeError("device status word set in the SmolLM2-shaped stack")
    return {"tokens": M, "rank": r, "layers": c["layers"], "ms_per_step": ms_g, "TFLOP/s": flops / ms_g / 1e9,
            "frac_bf16_burst": flops / ms_g / 1e9 / tc, "launches_per_step": launches,
            "single_calls": {"ms_per_step": ms_s, "TFLOP/s": flops / ms_s / 1e9},
            "flops_per_step": flops,
            "timing": "one step as a CUDA graph, L2 flushed before each replay, launch included"}


def sweep(dev, stream):
    """The workloads besides the bench line, timed through the C ABI (one JSON line each):
    the small-M forward of the Llama-3-8B-shaped matrices (GB/s of the bytes a forward must
    move: stored weight, fp32 adapters, activations), the SmolLM2-shaped 30-layer QLoRA stack
    (TFLOP/s) and the 1-D quantize / dequantize sizes (GB/s)."""
    import torch
    from bit_nf4_quantized_gb300 import binding as bq
    from bit_nf4_quantized_gb300 import workloads as wl
    lib = bq.load()
    pk, pk_src = peaks()
    hbm, tc = float(pk["hbm_gbs"]), float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)

    def emit(d):
        d["peaks"] = pk_src
        print(json.dumps(d), flush=True)

    # small-M forward of the 7 projections of one layer: the batched call (one T launch and one
    # weight pass for the whole layer) and the 7 single calls, each as one timed graph
    c = wl.W4
    r, Ms = c["r"], c["Ms"]
    mmax = max(Ms)
    shapes = [(N, K) for _, N, K in c["shapes"]]
    need = max(max(max(lib.qlora_fwd_workspace_bytes(m, N, K, r, 1) for N, K in shapes),
                   bq.qlora_fwd_batch_workspace_bytes(m, shapes, r)) for m in Ms)
    ws = torch.empty(max(16, need), dtype=torch.uint8, device=dev)
    projs = []
    for i, (_, N, K) in enumerate(c["shapes"]):
        seed = wl.seed_for(4, 100 * i)
        q = bq.nf4_quantize(wl.device_student_t((N, K), 5, 0.02, seed, dev, torch.bfloat16), True)
        projs.append(dict(N=N, K=K, q=q,
                          A=wl.device_normal((r, K), 1.0 / r, seed + 3, dev, torch.float32),
                          B=wl.device_normal((N, r), 0.01, seed + 4, dev, torch.float32),
                          x=wl.device_normal((mmax, K), 1.0, seed + 1, dev, torch.bfloat16),
                          y=torch.empty((mmax, N), dtype=torch.bfloat16, device=dev),
                          T=torch.empty((mmax, r), dtype=torch.float32, device=dev)))
    weight_bytes = sum(lib.nf4_packed_bytes(p["N"] * p["K"], 1) for p in projs)
    for m in Ms:
        items = [dict(x=p["x"][:m], W=p["q"], A=p["A"], B=p["B"], alpha=c["alpha"], y=p["y"][:m], T=p["T"][:m])
                 for p in projs]

        def batched():
            bq.qlora_linear_fwd_batch(items, workspace=ws)

        def single(m=m):
            for p in projs:
                bq.qlora_linear_fwd(p["x"][:m], p["q"], p["A"], p["B"], c["alpha"], y=p["y"][:m], T=p["T"][:m],
                                    workspace=ws)
        ms_b = graph_ms(batched, dev, stream, flush, reps=20)
        ms_s = graph_ms(single, dev, stream, flush, reps=20)
        nbytes = weight_bytes + sum(4 * r * (p["N"] + p["K"]) + 2 * m * (p["N"] + p["K"]) for p in projs)
        emit({"sweep": "small-M forward, 7 Llama-3-8B-shaped projections", "tokens": m, "rank": r,
              "ms_per_layer_batched": ms_b, "ms_per_layer_single_calls": ms_s,
              "weight_GB/s_batched": weight_bytes / ms_b / 1e6, "frac_hbm_batched": weight_bytes / ms_b / 1e6 / hbm,
              "GB/s_batched": nbytes / ms_b / 1e6, "GB/s_single_calls": nbytes / ms_s / 1e6,
              "weight_bytes_per_layer": weight_bytes, "bytes_per_layer": nbytes})
    del projs, ws

    # SmolLM2-shaped stack: QLoRA forward + backward on q and v of 30 layers
    st2 = measure_smollm2(dev, lambda fn: graph_ms(fn, dev, stream, flush), tc)
    emit(dict({"sweep": "SmolLM2-shaped stack, QLoRA q and v of 30 layers, fwd+bwd"}, **st2))

    # 1-D quantize (fp32 input) and dequantize (fp32 output)
    for n in wl.W5["sizes"]:
        x = wl.device_normal((n,), wl.W5["std"], wl.seed_for(5, 1), dev, torch.float32)
        q = bq.Nf4Tensor.empty((n,), True, dev)
        wsq = torch.empty(max(16, lib.nf4_quantize_workspace_bytes(n, 1)), dtype=torch.uint8, device=dev)
        y = torch.empty(n, dtype=torch.float32, device=dev)
        q_ms = graph_ms(lambda: bq.nf4_quantize(x, True, out=q, workspace=wsq), dev, stream, flush, reps=5)
        d_ms = graph_ms(lambda: bq.nf4_dequantize(q, out=y), dev, stream, flush, reps=5)
        stored = lib.nf4_packed_bytes(n, 1)
        emit({"sweep": "1-D NF4 double quant, fp32", "numel": n,
              "quantize_GB/s": (4 * n + stored + 4) / q_ms / 1e6, "dequantize_GB/s": (stored + 4 * n) / d_ms / 1e6,
              "quantize_frac_hbm": (4 * n + stored + 4) / q_ms / 1e6 / hbm,
              "dequantize_frac_hbm": (stored + 4 * n) / d_ms / 1e6 / hbm, "quantize_ms": q_ms, "dequantize_ms": d_ms})
        del x, q, wsq, y
    if bq.device_status() != bq.NF4_OK:
        raise RuntimeError("device status word set during the sweep")
    return 0


def profile_case(args):
    """Fixed workloads for ncu captures (commands in profiles/)."""
    import torch
    from bit_nf4_quantized_gb300 import binding as bq
    from bit_nf4_quantized_gb300 import workloads as wl
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    if args.profile_case == "gate_linear":
        c = wl.W3
        N, K = dict((n, (a, b)) for n, a, b in c["shapes"])["gate_proj"]
        M, r = c["M"], c["r"]
        w = wl.device_student_t((N, K), c["t_df"], c["w_scale"], wl.seed_for(3, 400), dev, torch.bfloat16)
        x = wl.device_normal((M, K), 1.0, wl.seed_for(3, 401), dev, torch.bfloat16)
        dy = wl.device_normal((M, N), 1.0, wl.seed_for(3, 402), dev, torch.bfloat16)
        A = wl.device_normal((r, K), 1.0 / r, wl.seed_for(3, 403), dev, torch.float32)
        B = wl.device_normal((N, r), 0.01, wl.seed_for(3, 404), dev, torch.float32)
        q = bq.nf4_quantize(w, True)
        bq.nf4_quantize(w, True, out=q)
        deq = bq.nf4_dequantize(q, torch.bfloat16)
        bq.nf4_dequantize(q, out=deq)
        for _ in range(3):
            y, T = bq.qlora_linear_fwd(x, q, A, B, c["alpha"])
        for _ in range(3):
            bq.qlora_linear_bwd(dy, x, T, q, A, B, c["alpha"])
    elif args.profile_case == "smollm2":
        # two SmolLM2-shaped layers (q and v share x, M = 512, r = 16): per layer one grouped forward
        # and one grouped backward, three times
        c = wl.W2
        M, r = c["M"], c["r"]
        targets = [(N, K) for n, N, K in c["shapes"] if n in c["targets"]]
        x = wl.device_normal((M, targets[0][1]), 1.0, wl.seed_for(2, 1), dev, torch.bfloat16)
        mats = []
        for layer in range(2):
            for j, (N, K) in enumerate(targets):
                seed = wl.seed_for(2, 1000 + 10 * (layer * 2 + j))
                q = bq.nf4_quantize(wl.device_normal((N, K), 0.02, seed, dev, torch.bfloat16), True)
                mats.append(dict(W=q, A=wl.device_normal((r, K), 1.0 / r, seed + 3, dev, torch.float32),
                                 B=wl.device_normal((N, r), 0.01, seed + 4, dev, torch.float32),
                                 dy=wl.device_normal((M, N), 1.0, seed + 2, dev, torch.bfloat16)))
        for _ in range(3):
            for layer in range(2):
                group = mats[2 * layer:2 * layer + 2]
                outs = bq.qlora_linear_fwd_batch([dict(x=x, W=m["W"], A=m["A"], B=m["B"], alpha=c["alpha"])
                                                  for m in group])
                bq.qlora_linear_bwd_batch([dict(dy=m["dy"], x=x, T=o[1], W=m["W"], A=m["A"], B=m["B"],
                                                alpha=c["alpha"]) for m, o in zip(group, outs)])
    elif args.profile_case == "small_m":
        c = wl.W4
        M = args.tokens
        items = []
        for i, (_, N, K) in enumerate(c["shapes"]):
            seed = wl.seed_for(4, 100 * i)
            q = bq.nf4_quantize(wl.device_student_t((N, K), 5, 0.02, seed, dev, torch.bfloat16), True)
            items.append(dict(x=wl.device_normal((M, K), 1.0, seed + 1, dev, torch.bfloat16), W=q,
                              A=wl.device_normal((c["r"], K), 1.0 / c["r"], seed + 3, dev, torch.float32),
                              B=wl.device_normal((N, c["r"]), 0.01, seed + 4, dev, torch.float32), alpha=c["alpha"]))
        for _ in range(4):
            bq.qlora_linear_fwd_batch(items)
    else:
        e = wl.W6
        table = random_stored_nf4((e["rows"], e["dim"]), wl.seed_for(6, 10), dev)
        g = torch.Generator(device=dev)
        g.manual_seed(wl.seed_for(6, 11))
        ids = torch.randint(0, e["rows"], (e["n_ids"],), generator=g, device=dev, dtype=torch.int64)
        for _ in range(2):
            bq.nf4_embedding_rows(table, ids, torch.bfloat16)
        del table
        m = wl.W7
        W = random_stored_nf4((m["N"], m["K"]), wl.seed_for(7, 20), dev)
        A = wl.device_normal((m["r"], m["K"]), 1.0 / m["r"], wl.seed_for(7, 21), dev, torch.float32)
        B = wl.device_normal((m["N"], m["r"]), 0.01, wl.seed_for(7, 22), dev, torch.float32)
        for _ in range(2):
            bq.nf4_merge_lora(W, A, B, m["alpha"])
    torch.cuda.synchronize()
    st = bq.device_status()
    print(json.dumps({"profile_case": args.profile_case, "device_status": st, "launches": bq.launch_count()}))
    return 0 if st == bq.NF4_OK else 1


def traffic_json(csv_path):
    """Per-launch DRAM traffic of the bf16 GEMM from an ncu CSV of one bench step, as the record
    bench.py reads (keyed to the SHA-256 of the GEMM source it was taken on)."""
    import csv
    import hashlib
    from bit_nf4_quantized_gb300 import workloads as wl
    rows = {}
    with open(csv_path) as f:
        for rec in csv.DictReader(line for line in f if line.startswith('"')):
            if "bf16_tc_gemm" not in rec.get("Kernel Name", ""):
                continue
            d = rows.setdefault(rec["ID"], {})
            v = float(rec["Metric Value"].replace(",", ""))
            unit = rec.get("Metric Unit", "")
            scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "ns": 1, "us": 1e3, "usecond": 1e3,
                     "nsecond": 1, "ms": 1e6}.get(unit, 1)
            d[rec["Metric Name"]] = v * scale
    launches = [rows[k] for k in sorted(rows, key=int)][-14:]
    names = [n for n, _, _ in wl.W3["shapes"]]
    rec = {"kernel": "bf16_tc_gemm", "workload": "one step of the Llama-3-8B-shaped layer (7 projections, M = 4096, r = 16)",
           "launches": {"fwd_gemm": [], "dx_gemm": []}}
    for i, d in enumerate(launches):   # the step's 7 forward GEMMs, then its 7 dX GEMMs
        kind = "fwd_gemm" if i < len(names) else "dx_gemm"
        rec["launches"][kind].append({"projection": names[i % len(names)].split("_")[0],
                                      "dram_bytes": int(d.get("dram__bytes_read.sum", 0) + d.get("dram__bytes_write.sum", 0)),
                                      "duration_ns": int(d.get("gpu__time_duration.sum", 0))})
    rec["per_launch_bytes"] = {k: int(sum(x["dram_bytes"] for x in v) / max(1, len(v))) for k, v in rec["launches"].items()}
    with open(os.path.join(ROOT, "bit_nf4_quantized_gb300", "csrc", "linear_tc.cu"), "rb") as f:
        rec["source_sha256"] = hashlib.sha256(f.read()).hexdigest()
    print(json.dumps(rec, indent=1))
    return 0


def main():
    args = parse()
    if args.cpu_sample_worker is not None:
        return cpu_sample_worker(args.cpu_sample_worker)
    if args.traffic_json:
        return traffic_json(args.traffic_json)
    if args.cpu_plan_worker:
        return cpu_plan_worker(args.cpu_plan_worker, args.cpu_plan_max_log2)
    if args.cpu_plan:
        return cpu_plan(args)
    if args.profile_case:
        return profile_case(args)
    rank, world, local = dist_setup()
    if args.impl == "reference":
        return reference_arm(args, rank, world)
    if args.sweep:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        torch.cuda.set_device(local)
        dev = torch.device("cuda", local)
        return sweep(dev, torch.cuda.current_stream(dev)) if rank == 0 else 0

    # the oracle sample runs before the first CUDA call in this process
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline()

    import torch
    from bit_nf4_quantized_gb300 import binding
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    layer = Layer(dev, only=args.only)
    pk, pk_src = peaks()
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.5)
    for _ in range(max(args.warmup, 3)):
        layer.step()
    torch.cuda.synchronize(dev)
    if binding.device_status() != binding.NF4_OK:
        raise RuntimeError("device status word set during warm-up")

    # one step (every kernel of the path, the same arguments) captured into a CUDA graph
    # and replayed: what a training loop does to take host launch overhead off the GPU
    graph = torch.cuda.CUDAGraph()
    launches0 = binding.launch_count()
    with torch.cuda.graph(graph):
        layer.step()
    per_step_launches = binding.launch_count() - launches0
    graph.replay()
    torch.cuda.synchronize(dev)
    if binding.device_status() != binding.NF4_OK:
        raise RuntimeError("device status word set by the captured step")
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    ms = time_steps(graph.replay, args.steps, stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    barrier(world)
    launches = per_step_launches * args.steps
    # per-phase breakdown (the dominant kernel's roofline): the same steps again with the
    # library's per-launch CUDA events on, outside the timed region above
    binding.timing_enable(True)
    for k in range(6):
        binding.timing_read(k, reset=True)
    for _ in range(args.steps):
        layer.step()
    torch.cuda.synchronize(dev)
    binding.timing_enable(False)
    sampler.stop()
    kinds = {name: binding.timing_read(k, reset=True) for k, name in
             enumerate(("quantize", "dequantize", "fwd_gemm", "dx_gemm", "adapter", "weight_decode"))}
    ms_max = max_over_ranks(ms, world)

    M, r = layer.M, layer.r
    flops = layer_flops(layer.shapes, M, r)
    value = world * flops * args.steps / (ms_max / 1e3) / 1e12
    # dominant kernel: the base contraction kind with the larger share of time
    fwd_f = sum(2 * M * N * K + 2 * M * N * r for _, N, K in layer.shapes)
    dx_f = sum(2 * M * N * K + 2 * M * K * r for _, N, K in layer.shapes)
    dom = "fwd_gemm" if kinds["fwd_gemm"][0] >= kinds["dx_gemm"][0] else "dx_gemm"
    dom_ms, dom_n = kinds[dom]
    dom_flops = (fwd_f if dom == "fwd_gemm" else dx_f) * args.steps
    achieved = dom_flops / (dom_ms / 1e3) / 1e12 if dom_ms > 0 else 0.0
    # a GEMM launch lasts well under a millisecond: the burst cuBLAS figure is its peak; the
    # sustained (seconds-long, power-capped) figure is reported beside it
    peak = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sus = float(pk.get("bf16_tflops_sustained", peak))
    nel = sum(N * K for _, N, K in layer.shapes)
    deq_bytes = nel * 2 + sum(binding.load().nf4_packed_bytes(N * K, 1) for _, N, K in layer.shapes)
    deq_ms, deq_n = kinds["dequantize"]
    deq_gbs = deq_bytes * args.steps / (deq_ms / 1e3) / 1e9 if deq_ms > 0 else 0.0
    q_ms, _ = kinds["quantize"]
    q_bytes = nel * 2 + sum(binding.load().nf4_packed_bytes(N * K, 1) + 4 for _, N, K in layer.shapes)
    q_gbs = q_bytes * args.steps / (q_ms / 1e3) / 1e9 if q_ms > 0 else 0.0
    hbm = float(pk["hbm_gbs"])
    clocks = sampler.summary(t0, t1)

    # the quantize and dequantize rows on their own: each row's 7 calls (same kernels and
    # arguments as in the step) captured as a graph and replayed, L2 flushed between replays
    # (a 256 MB write outside the timed intervals)
    from bit_nf4_quantized_gb300 import binding as bq
    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)

    def row_ms(fn, reps=10):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        g.replay()
        torch.cuda.synchronize(dev)
        total = 0.0
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            total += a.elapsed_time(b)
        return total / reps

    q_row_ms = row_ms(layer.quantize_all)
    q_single_ms = row_ms(lambda: [bq.nf4_quantize(p["w"], True, out=p["q"], workspace=layer.ws_q) for p in layer.proj])
    # the dequantize row: the layer's 7 weights in one nf4_dequantize_batch call (7 outputs), and
    # as 7 nf4_dequantize calls into the step's one buffer
    deq_outs = [torch.empty((p["N"], p["K"]), dtype=torch.bfloat16, device=dev) for p in layer.proj]
    d_row_ms = row_ms(lambda: bq.nf4_dequantize_batch([(p["q"], o) for p, o in zip(layer.proj, deq_outs)]))
    d_single_ms = row_ms(lambda: [bq.nf4_dequantize(p["q"], out=layer.deq[:p["N"] * p["K"]].view(p["N"], p["K"]))
                                  for p in layer.proj])
    del deq_outs
    deq_row_gbs = deq_bytes / (d_row_ms / 1e3) / 1e9
    q_row_gbs = q_bytes / (q_row_ms / 1e3) / 1e9
    export_rows = measure_export_rows(dev, row_ms, hbm)
    no_dq = measure_no_double_quant(layer, row_ms)
    small_m = measure_small_m(layer, row_ms, hbm)
    f16_profile = measure_f16_profile(layer, row_ms)
    fp32_576 = measure_fp32_576(dev, row_ms)
    smollm2 = measure_smollm2(dev, row_ms, peak)
    # the same step as one graph with L2 flushed before it: all 7 weights decoded first (the
    # headline's step), each decoded right before its projection, and the NF4-input calls, which
    # decode the weight once per call
    first_ms = row_ms(layer.step, reps=5)
    layer.grouped = False
    single_ms = row_ms(layer.step, reps=5)
    layer.decode_batch = False
    once_ms = row_ms(layer.step, reps=5)
    layer.decode_once = False
    per_call_ms = row_ms(layer.step, reps=5)
    layer.decode_once = True
    layer.decode_batch = True
    layer.grouped = True
    step_variants = {"grouped": {"ms_per_step": first_ms, "TFLOP/s": flops / (first_ms / 1e3) / 1e12},
                     "single_calls": {"ms_per_step": single_ms, "TFLOP/s": flops / (single_ms / 1e3) / 1e12},
                     "decode_before_each": {"ms_per_step": once_ms, "TFLOP/s": flops / (once_ms / 1e3) / 1e12},
                     "decode_per_call": {"ms_per_step": per_call_ms, "TFLOP/s": flops / (per_call_ms / 1e3) / 1e12},
                     "timing": "one step as a graph, L2 flushed before each replay, launch included",
                     "what": "grouped = the headline step; single_calls = the same decode, then per projection "
                             "qlora_linear_fwd_w16 / qlora_linear_bwd_w16; decode_before_each = each weight "
                             "decoded right before its single calls; decode_per_call = the NF4-input calls"}

    e2e = None
    if not args.no_e2e:
        # each projection's inputs (bf16 master weight, dY; a shared x once) come from pinned host
        # memory and its dA, dB go back; the copies run on two copy streams (each tensor in halves,
        # one per copy engine) ahead of the compute; each set of projections that reads one x runs
        # the headline's calls (quantize batch, dequantize batch, grouped forward and backward)
        # once its own inputs are in
        local_cpus = gpu_local_cpus(dev)
        saved_affinity = os.sched_getaffinity(0)
        if local_cpus:
            os.sched_setaffinity(0, local_cpus)
        groups = layer.x_groups()
        dev_in = [[t for i in idx for t in ([layer.proj[i]["w"], layer.proj[i]["dy"]] +
                                            ([layer.proj[i]["x"]] if layer.x_first[layer.proj[i]["x_of"]] == i
                                             else []))] for idx in groups]
        dev_out = [[t for i in idx for t in layer.results_of(layer.proj[i])] for idx in groups]
        host_in = [[t.cpu().pin_memory() for t in ts] for ts in dev_in]
        host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ts] for ts in dev_out]
        h2d = sum(t.numel() * t.element_size() for hs in host_in for t in hs)
        d2h = sum(t.numel() * t.element_size() for hs in host_out for t in hs)
        copy_streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
        ready = [[torch.cuda.Event() for _ in copy_streams] for _ in groups]
        done = [torch.cuda.Event() for _ in groups]   # the set's compute and read-back issued

        def e2e_step():
            for g in range(len(groups)):
                for c, cs in enumerate(copy_streams):
                    with torch.cuda.stream(cs):
                        cs.wait_event(done[g])   # the previous step has finished with these buffers
                        for h, d in zip(host_in[g], dev_in[g]):
                            half = (h.shape[0] + 1) // 2
                            lo, hi = (0, half) if c == 0 else (half, h.shape[0])
                            d[lo:hi].copy_(h[lo:hi], non_blocking=True)
                        ready[g][c].record(cs)
            for g, idx in enumerate(groups):
                for ev in ready[g]:
                    stream.wait_event(ev)
                layer.run_group(idx)
                for h, d in zip(host_out[g], dev_out[g]):
                    h.copy_(d, non_blocking=True)
                done[g].record(stream)

        def time_e2e(steps):
            # the copy streams start after the start event; each step's copies then wait only
            # for the previous step's use of the same buffers, so copies run back to back
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            for cs in copy_streams:
                cs.wait_event(start)
            for _ in range(steps):
                e2e_step()
            end.record(stream)
            end.synchronize()
            return start.elapsed_time(end)

        e2e_step()
        torch.cuda.synchronize(dev)
        barrier(world)
        e_steps = max(3, args.steps // 3)
        e_ms = max_over_ranks(time_e2e(e_steps), world)
        barrier(world)
        os.sched_setaffinity(0, saved_affinity)
        e2e = {"value": world * flops * e_steps / (e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
               "host_threads": (f"held on the GPU's {len(local_cpus)} local CPUs while the pinned "
                                "buffers are allocated and the steps are issued") if local_cpus
                               else "not held (no local CPU list for this GPU)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAME, "tokens": M, "rank": r, "alpha": layer.alpha,
                       "targets": [n for n, _, _ in layer.shapes], "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2: each step touches ~1.5 GB of distinct buffers",
                       "step": "nf4_quantize_batch of the 7 bf16 masters, nf4_dequantize_batch of the 7 "
                               "quantized weights (bf16), then one qlora_linear_fwd_batch and one "
                               "qlora_linear_bwd_batch over the 7 projections reading their decoded weights; q, k, v "
                               "read one x and gate, up another (as in a transformer layer), and each such set "
                               "shares one T pass and one dA pass (key step_variants also times per-projection "
                               "single calls)",
                       "launch": "one step captured as a CUDA graph, replayed per timed step"},
            "gpu_launches": launches,
            "phases_ms_per_step": {k: v[0] / args.steps for k, v in kinds.items()},
            "roofline": {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak if peak else None, "traffic": gemm_traffic(dom),
                         "peak_source": f"{pk_src} bf16_tflops (cuBLAS bf16 GEMM, burst)", "launches": dom_n,
                         "sustained_peak": peak_sus, "frac_of_sustained": achieved / peak_sus if peak_sus else None,
                         "clock_normalised": clock_normalised(achieved, clocks, peak_sus, pk)},
            "dequant": {"GB/s": deq_row_gbs, "frac": deq_row_gbs / hbm, "peak_gbs": hbm,
                        "bytes_per_step": deq_bytes, "ms_per_step": d_row_ms,
                        "timing": "the layer's 7 weights in one nf4_dequantize_batch call as a graph, L2 flushed "
                                  "between replays",
                        "single_calls": {"ms_per_step": d_single_ms, "GB/s": deq_bytes / (d_single_ms / 1e3) / 1e9,
                                         "frac": deq_bytes / (d_single_ms / 1e3) / 1e9 / hbm,
                                         "timing": "the 7 nf4_dequantize calls as one graph"},
                        "GB/s_in_step_events": deq_gbs, "launches": deq_n},
            "quantize": {"GB/s": q_row_gbs, "frac": q_row_gbs / hbm, "bytes_per_step": q_bytes,
                         "ms_per_step": q_row_ms,
                         "timing": "the layer's 7 weights in one nf4_quantize_batch call as a graph, L2 flushed "
                                   "between replays",
                         "GB/s_in_step_events": q_gbs,
                         "single_calls": {"ms_per_step": q_single_ms, "GB/s": q_bytes / (q_single_ms / 1e3) / 1e9,
                                          "frac": q_bytes / (q_single_ms / 1e3) / 1e9 / hbm,
                                          "timing": "the 7 nf4_quantize calls as one graph"}},
            "step_variants": step_variants,
            "no_double_quant": no_dq,
            "small_m_forward": small_m,
            "f16_profile": f16_profile,
            "fp32_576": fp32_576,
            "smollm2_stack": smollm2,
            "embedding": export_rows["embedding"],
            "merge": export_rows["merge"],
            "clocks": clocks,
            "e2e": e2e,
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
