"""Benchmark of the fused FFN (and its decode / large / MoE workloads).

python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME|all] [--impl reference]

By default (--config all) it measures five workloads one after the other --
the tiny, prefill, decode, large and MoE FFNs -- and prints ONE line: the
headline fields are the prefill FFN's, `configs` holds every workload's
entry (value, roofline, end-to-end figures, clocks, CPU oracle baseline),
`small_m` summarises the decode workload (weight GB/s) and `large_m` the
large one (TFLOP/s).  --config NAME measures one workload.

A step is one ffn_forward (or moe_ffn_forward) call over one batch of
synthetic input resident in HBM.  Timing: W untimed warm-up steps, then K
steps, each bracketed by CUDA events on the launching stream; when a step's
inputs are under twice the L2 (129 MB), a 256 MiB write between steps so that
L2 holds nothing of the previous step (larger inputs stream through it);
a barrier + device synchronisation on both sides of the timed block; the max
over ranks.  Under torchrun every rank runs its own replica of the workload
(the FFN has no data-path exchange: weak scaling, no collective but the
timing barrier and max).

Printed (rank 0): one JSON line with the metric, the roofline of the dominant
kernel (its own CUDA-event time inside the timed steps), the end-to-end
number through the public API with pinned host buffers (inputs copied in,
result copied out inside the timed region), the clocks sampled during the
timed region, and the CPU oracle timed on a bounded sample of the workload
(rank 0, N = 1).  --impl reference times that oracle as the reference arm.
"""
import argparse
import hashlib
import re
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

# ----------------------------------------------------------------- workloads
CONFIGS = {
    "tiny": dict(kind="ffn", M=64, N=256, O=1024, P=256, act1="gelu_tanh", act2="none",
                 label="tiny dense FFN M=64 N=256 O=1024 P=256, GELU-tanh"),
    "prefill": dict(kind="ffn", M=4096, N=4096, O=16384, P=4096, act1="gelu_tanh", act2="none",
                    label="prefill FFN M=4096 N=4096 O=16384 P=4096, GELU-tanh"),
    "decode": dict(kind="ffn", M=16, N=8192, O=28672, P=8192, act1="relu", act2="none",
                   label="decode FFN M=16 N=8192 O=28672 P=8192, ReLU"),
    "large": dict(kind="ffn", M=16384, N=8192, O=28672, P=8192, act1="gelu_tanh", act2="relu",
                  label="large prefill FFN M=16384 N=8192 O=28672 P=8192, GELU-tanh + ReLU"),
    "large_m2048": dict(kind="ffn", M=2048, N=8192, O=28672, P=8192, act1="gelu_tanh", act2="relu",
                        label="large-FFN dimensions at 2048 rows (M=2048 N=8192 O=28672 P=8192, GELU-tanh + ReLU): "
                              "the engine on the large FFN's weights with a footprint small enough for a full ncu "
                              "capture"),
    "moe": dict(kind="moe", M=8192, N=4096, O=14336, P=4096, E=8, k=2, act1="gelu_tanh", act2="none",
                label="MoE FFN T=8192 N=4096 E=8 O=14336 P=4096, softmax top-2, GELU-tanh"),
    "swiglu": dict(kind="glu", M=4096, N=4096, O=14336, P=4096, act1="silu", act2="none",
                   label="SwiGLU FFN (Llama 3 8B shape) M=4096 N=4096 O=14336 P=4096, "
                         "Y = (SiLU(X W1) * (X W3)) W2, no biases"),
    "swiglu_decode": dict(kind="glu", M=16, N=4096, O=14336, P=4096, act1="silu", act2="none",
                          label="SwiGLU FFN decode (Llama 3 8B shape) M=16 N=4096 O=14336 P=4096"),
    "batch128": dict(kind="ffn", M=128, N=4096, O=14336, P=4096, act1="gelu_tanh", act2="none",
                     label="batched decode FFN (Llama 3 8B dims) M=128 N=4096 O=14336 P=4096, GELU-tanh"),
    "swiglu_batch128": dict(kind="glu", M=128, N=4096, O=14336, P=4096, act1="silu", act2="none",
                            label="SwiGLU FFN batched decode (Llama 3 8B shape) M=128 N=4096 O=14336 P=4096"),
    "moe_swiglu": dict(kind="moe", glu=True, M=8192, N=4096, O=14336, P=4096, E=8, k=2, act1="silu",
                       act2="none",
                       label="MoE FFN with SwiGLU experts (Mixtral-class) T=8192 N=4096 E=8 O=14336 P=4096, "
                             "softmax top-2"),
    "moe_moderate": dict(kind="moe", M=8192, N=4096, O=14336, P=4096, E=8, k=2, act1="gelu_tanh",
                         act2="none", router="moderate",
                         label="MoE FFN T=8192 N=4096 E=8 O=14336 P=4096, softmax top-2, GELU-tanh, "
                               "moderately skewed router (logit offsets -ln(1+e))"),
    "moe_stress": dict(kind="moe", M=8192, N=4096, O=14336, P=4096, E=8, k=2, act1="gelu_tanh",
                       act2="none", router="stress",
                       label="MoE FFN T=8192 N=4096 E=8 O=14336 P=4096, softmax top-2, GELU-tanh, "
                             "stress-skewed router (expert 0 in ~98% of tokens)"),
}
# The default run measures these five workloads (the tiny, prefill, decode,
# large and MoE FFNs) and prints one line whose headline is the prefill FFN;
# --config NAME measures one workload.
SUITE = ("tiny", "prefill", "decode", "large", "moe")
HEADLINE = "prefill"
DEFAULT = "all"
FFN_PATHS = {"auto": 0, "fused": 1, "decode": 2, "two": 3, "reduce": 4, "b2b": 5, "stream": 6}
FLUSH_BYTES = 256 << 20
SPEC_BF16_TFLOPS = 2250.0   # GB300 dense bf16 (NVIDIA's 2:4-sparse figures are twice this)
SPEC_HBM_GBS = 8000.0       # GB300 HBM3e

# Dominant kernel of each workload (for the ncu traffic record).
DECODE_MAX_M = 32   # rows up to which ffn_forward / ffn_glu_forward stream the weights with mma.sync
STREAM_MAX_M = 128  # ... and then with tcgen05 MMAs
KERNEL = {"tiny": "decode_kernel", "prefill": "engine_kernel", "large": "engine_kernel",
          "swiglu": "engine_kernel", "swiglu_decode": "decode_kernel", "moe": "engine_kernel", "moe_swiglu": "engine_kernel", "moe_moderate": "engine_kernel", "moe_stress": "engine_kernel",
          "decode": "decode_kernel", "batch128": "wstream_kernel", "swiglu_batch128": "wstream_kernel"}
# Sources a kernel's DRAM traffic depends on: its own code and the host code
# that builds its tensor maps (box shapes, L2 promotion).
KERNEL_SOURCES = {
    "engine_kernel": ["engine.cuh", "common.cuh", "ptx.cuh", "schedule.h", "engine_dense.cu",
                      "engine_grouped.cu", "api.cu"],
    "decode_kernel": ["decode.cu", "decode.cuh", "common.cuh", "ptx.cuh", "api.cu"],
    "reduce_kernel": ["reduce.cuh", "reduce_params.cuh", "engine.cuh", "common.cuh", "ptx.cuh", "engine_reduce.cu",
                      "api.cu"],
    "b2b_kernel": ["reduce.cuh", "reduce_params.cuh", "engine.cuh", "common.cuh", "ptx.cuh", "engine_reduce.cu",
                   "api.cu"],
    "wstream_kernel": ["wstream.cu", "wstream.cuh", "common.cuh", "ptx.cuh", "api.cu"],
}


def dominant_kernel(config, ffn_path="auto"):
    """The kernel whose launches the roofline times for this workload."""
    if ffn_path == "reduce" and CONFIGS[config]["kind"] == "ffn":
        return "reduce_kernel"
    if ffn_path == "b2b" and CONFIGS[config]["kind"] == "ffn":
        return "b2b_kernel"
    if ffn_path == "decode" and CONFIGS[config]["kind"] in ("ffn", "glu"):
        return "decode_kernel"
    if ffn_path == "stream" and CONFIGS[config]["kind"] in ("ffn", "glu"):
        return "wstream_kernel"
    if ffn_path in ("fused", "two"):
        return "engine_kernel"
    cfg = CONFIGS[config]
    if cfg["kind"] in ("ffn", "glu"):
        # the library's own choice (for the workloads defined here): the mma.sync
        # stream up to 32 rows, the tensor-core stream to 128, the engine above
        if cfg["M"] <= DECODE_MAX_M:
            return "decode_kernel"
        return "wstream_kernel" if cfg["M"] <= STREAM_MAX_M else "engine_kernel"
    return KERNEL[config]


def flops(cfg):
    """Algorithmic FLOPs of one step: 2*rows*O*(N+P), routed rows for MoE;
    2*M*O*(2N+P) for the gated FFN (two input products)."""
    rows = cfg["M"] * cfg.get("k", 1)
    n_in = 2 * cfg["N"] if (cfg["kind"] == "glu" or cfg.get("glu")) else cfg["N"]
    return 2.0 * rows * cfg["O"] * (n_in + cfg["P"])


def weight_bytes(cfg):
    """Bytes the decode step must move: W1, W2, X, Y, b1, b2 (bf16); the gated
    FFN reads W1, W3, W2 and has no biases."""
    M, N, O, P = cfg["M"], cfg["N"], cfg["O"], cfg["P"]
    if cfg["kind"] == "glu":
        return 2.0 * (2 * N * O + O * P + M * N + M * P)
    return 2.0 * (N * O + O * P + M * N + M * P + O + P)


def is_hbm_bound(cfg):
    # the weight streams: M up to 128 rows, below the ridge (2 M FLOP per weight byte pair)
    return cfg["kind"] in ("ffn", "glu") and cfg["M"] <= STREAM_MAX_M


def metric_of(cfg):
    if is_hbm_bound(cfg):
        return "fused FFN weight-stream bandwidth (small M)", "GB/s"
    return "fused FFN throughput (large M)", "TFLOP/s"


def rate(cfg, seconds):
    if is_hbm_bound(cfg):
        return weight_bytes(cfg) / seconds / 1e9
    return flops(cfg) / seconds / 1e12


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["bf16_tflops"], d["hbm_gbs"], "measured"
    except Exception:
        return 1900.0, 6800.0, "fallback"


def sustained_bf16_peak():
    """cuBLAS bf16 throughput held for seconds under the power cap (context
    for long runs of a tensor-bound kernel), or None."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        return None


def _code_only(text):
    """Source text without comments and with whitespace runs collapsed, so that
    a record taken on a kernel stays valid across comment-only edits."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_sha(kernel):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "transformer_ffn_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(config, kernel=None):
    """DRAM bytes per launch from the committed ncu record, if it was taken
    on the kernel source as it is now (else None)."""
    kernel = kernel or KERNEL[config]
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_sha(kernel)
    for line in open(path):
        if line.startswith("#") or "=" not in line:
            continue
        kv = dict(p.split("=", 1) for p in line.split())
        if kv.get("config") == config and kv.get("kernel") == kernel and kv.get("src_sha") == want:
            return float(kv["dram_bytes_per_launch"])
    return None


# -------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 20 ms, each sample stamped,
    so that the median and the reasons come from the samples taken inside the
    timed region (mark() brackets it)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 20

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None
        self.window = [None, None]

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.1)   # the first samples arrive before the timed region starts

    def mark(self, which):
        self.window[0 if which == "start" else 1] = time.time()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        return summarize_clocks(self.lines, self.window, self.INTERVAL_MS)


def summarize_clocks(lines, window, interval_ms):
    """Median SM clock, max clock and active throttle reasons of the samples
    (nvidia-smi csv lines: timestamp, index, clocks.sm, clocks.max.sm, power,
    reasons.active, hw_slowdown, hw_thermal_slowdown, sw_thermal_slowdown,
    sw_power_cap) taken inside window = [t0, t1] (host epoch seconds, one
    interval of slack on each side); the sample nearest the window when none
    falls inside it."""
    import datetime
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    samples = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            samples.append((ts, float(parts[2]), float(parts[3]),
                            {n for n, v in zip(names, parts[6:10]) if v.lower() == "active"}))
        except ValueError:
            continue
    if not samples:
        return None
    t0, t1 = window
    slack = interval_ms / 1e3
    inside = [x for x in samples if t0 is not None and t1 is not None and t0 - slack <= x[0] <= t1 + slack]
    where = "timed region"
    if not inside:
        ref = t0 if t0 is not None else samples[0][0]
        inside = [min(samples, key=lambda x: abs(x[0] - ref))]
        where = "nearest sample to the timed region"
    reasons = set()
    for x in inside:
        reasons |= x[3]
    return {"sm_mhz": statistics.median(x[1] for x in inside), "sm_max_mhz": max(x[2] for x in samples),
            "reasons": sorted(reasons), "samples": len(inside), "interval_ms": interval_ms, "from": where}


# ------------------------------------------------------------------- helpers
def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def make_inputs(cfg, device, seed=0):
    from transformer_ffn_gb300 import synth
    if cfg["kind"] == "glu":
        return synth.glu_inputs(cfg["M"], cfg["N"], cfg["O"], cfg["P"], seed=seed, device=device)
    if cfg["kind"] == "moe" and cfg.get("glu"):
        return synth.moe_glu_inputs(cfg["M"], cfg["N"], cfg["O"], cfg["P"], cfg["E"], seed=seed, device=device,
                                    router=cfg.get("router", "balanced"))
    if cfg["kind"] == "moe":
        return synth.moe_inputs(cfg["M"], cfg["N"], cfg["O"], cfg["P"], cfg["E"], seed=seed, device=device,
                                router=cfg.get("router", "balanced"))
    return synth.ffn_inputs(cfg["M"], cfg["N"], cfg["O"], cfg["P"], seed=seed, device=device)


def moe_call(cfg, inp, X, logits, out=None, routing=False, stream=None):
    """One MoE step through the library (gated experts when the workload has them)."""
    import transformer_ffn_gb300 as tffn
    if cfg.get("glu"):
        return tffn.moe_glu_forward(X, logits, cfg["k"], inp.W1, inp.W3, inp.W2, cfg["act1"], out=out,
                                    routing=routing, stream=stream)
    return tffn.moe_ffn_forward(X, logits, cfg["k"], inp.W1, inp.b1, inp.W2, inp.b2, cfg["act1"], cfg["act2"],
                                out=out, routing=routing, stream=stream)


def step_fn(cfg, inp, out, X=None):
    import transformer_ffn_gb300 as tffn
    X = inp.X if X is None else X
    if cfg["kind"] == "glu":
        return lambda: tffn.ffn_glu_forward(X, inp.W1, inp.W3, inp.W2, cfg["act1"], out=out)
    if cfg["kind"] == "moe":
        return lambda: moe_call(cfg, inp, X, inp.logits, out=out)
    return lambda: tffn.ffn_forward(X, inp.W1, inp.b1, inp.W2, inp.b2, cfg["act1"], cfg["act2"], out=out)


def run_e2e(cfg, inp, args, flush_buf, stream):
    """Mean seconds per step of the pipelined end-to-end loop, and the bytes
    copied host->device and device->host per step."""
    import torch
    import transformer_ffn_gb300 as tffn
    dev = inp.X.device
    moe = cfg["kind"] == "moe"
    X_host = inp.X.cpu().pin_memory()
    L_host = inp.logits.cpu().pin_memory() if moe else None
    Y_host = [torch.empty((cfg["M"], cfg["P"]), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    X_dev = [torch.empty_like(inp.X) for _ in range(2)]
    L_dev = [torch.empty_like(inp.logits) for _ in range(2)] if moe else None
    Y_dev = [torch.empty((cfg["M"], cfg["P"]), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    comp = stream
    ev = lambda: torch.cuda.Event()
    uploaded = [ev(), ev()]
    computed = [ev(), ev()]
    downloaded = [ev(), ev()]
    for e in computed + downloaded:
        e.record(comp)

    def step(i):
        b = i % 2
        with torch.cuda.stream(up):
            up.wait_event(computed[b])          # step i-2 no longer reads X_dev[b]
            X_dev[b].copy_(X_host, non_blocking=True)
            if moe:
                L_dev[b].copy_(L_host, non_blocking=True)
            uploaded[b].record(up)
        comp.wait_event(uploaded[b])
        comp.wait_event(downloaded[b])          # step i-2's result has left Y_dev[b]
        with torch.cuda.stream(comp):
            if moe:
                moe_call(cfg, inp, X_dev[b], L_dev[b], out=Y_dev[b], stream=comp)
            elif cfg["kind"] == "glu":
                tffn.ffn_glu_forward(X_dev[b], inp.W1, inp.W3, inp.W2, cfg["act1"], out=Y_dev[b], stream=comp)
            else:
                tffn.ffn_forward(X_dev[b], inp.W1, inp.b1, inp.W2, inp.b2, cfg["act1"], cfg["act2"],
                                 out=Y_dev[b], stream=comp)
        computed[b].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(computed[b])
            Y_host[b].copy_(Y_dev[b], non_blocking=True)
            downloaded[b].record(down)

    for i in range(max(2, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    if flush_buf is not None:
        flush_buf.zero_()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(up)
    for i in range(args.steps):
        step(i)
    end.record(down)
    torch.cuda.synchronize()
    tffn.check()
    h2d = X_host.numel() * 2 + (L_host.numel() * 4 if moe else 0)
    d2h = Y_host[0].numel() * 2
    return start.elapsed_time(end) / 1e3 / args.steps, h2d, d2h


# ----------------------------------------------------------------- GPU arm
def input_bytes(cfg):
    """Bytes of one step's inputs: activations, weights, biases (and logits)."""
    M, N, O, P = cfg["M"], cfg["N"], cfg["O"], cfg["P"]
    if cfg["kind"] == "glu":
        return 2 * (M * N + 2 * N * O + O * P)
    experts = cfg.get("E", 1)
    if cfg.get("glu"):
        b = 2 * M * N + experts * 2 * (2 * N * O + O * P)
    else:
        b = 2 * M * N + experts * 2 * (N * O + O * P + O + P)
    if cfg["kind"] == "moe":
        b += 4 * M * cfg["E"]
    return b


def l2_policy(cfg, dev):
    """Flush L2 between timed steps unless one step's inputs exceed twice its
    size (then no step can find the previous one's data in L2 anyway)."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    ib = input_bytes(cfg)
    if ib > 2 * l2:
        return False, (f"not flushed: each step's inputs ({ib / 2**20:.0f} MiB) exceed twice the "
                       f"L2 ({l2 / 2**20:.0f} MiB)")
    return True, f"flushed between steps ({FLUSH_BYTES >> 20} MiB write outside the step events)"


def time_steps(step, steps, flush_buf, stream):
    """Device time (s) of `steps` steps.  With an L2 flush between steps
    (flush_buf written outside the step events), each step is bracketed by
    its own pair of events and the per-step times are returned.  Without one,
    the steps run back to back between one pair of events (an event record
    between two kernels serialises them, which would add its own gap to every
    step) and the list holds the block's mean once per step."""
    import torch
    if flush_buf is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) / 1e3 / steps] * steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        flush_buf.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) / 1e3 for a, b in evs]


def run_e2e_latency(cfg, inp, steps, warmup, stream):
    """Per-call latency through the public API, one call at a time: upload the
    step's input from pinned host memory, run the FFN, download its result,
    synchronise; host wall clock around all four.  Returns the per-step
    seconds."""
    import torch
    import transformer_ffn_gb300 as tffn
    moe = cfg["kind"] == "moe"
    X_host = inp.X.cpu().pin_memory()
    L_host = inp.logits.cpu().pin_memory() if moe else None
    Y_host = torch.empty((cfg["M"], cfg["P"]), dtype=torch.bfloat16).pin_memory()
    X_dev = torch.empty_like(inp.X)
    L_dev = torch.empty_like(inp.logits) if moe else None
    Y_dev = torch.empty((cfg["M"], cfg["P"]), dtype=torch.bfloat16, device=inp.X.device)
    times = []
    for i in range(warmup + steps):
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            X_dev.copy_(X_host, non_blocking=True)
            if moe:
                L_dev.copy_(L_host, non_blocking=True)
            if moe:
                moe_call(cfg, inp, X_dev, L_dev, out=Y_dev, stream=stream)
            elif cfg["kind"] == "glu":
                tffn.ffn_glu_forward(X_dev, inp.W1, inp.W3, inp.W2, cfg["act1"], out=Y_dev, stream=stream)
            else:
                tffn.ffn_forward(X_dev, inp.W1, inp.b1, inp.W2, inp.b2, cfg["act1"], cfg["act2"], out=Y_dev,
                                 stream=stream)
            Y_host.copy_(Y_dev, non_blocking=True)
        stream.synchronize()
        if i >= warmup:
            times.append(time.perf_counter() - t0)
    tffn.check()
    return times


def run_unfused(cfg, inp, steps, warmup, stream):
    """Context comparator (bench only, never the library's path): the same
    dense or gated FFN as separate kernels -- cuBLAS GEMMs through
    torch.matmul and torch's elementwise bias / activation kernels, H kept in
    bf16 between the layers as the fused path keeps it.  Returns the mean
    seconds per step (one event pair around back-to-back steps)."""
    import torch
    import torch.nn.functional as F
    acts = {"none": lambda x: x, "relu": F.relu, "gelu_tanh": lambda x: F.gelu(x, approximate="tanh"),
            "silu": F.silu}
    a1, a2 = acts[cfg["act1"]], acts[cfg["act2"]]
    X = inp.X
    if cfg["kind"] == "glu":
        def step():
            H = a1(X @ inp.W1) * (X @ inp.W3)
            return H @ inp.W2
    else:
        def step():
            H = a1(torch.addmm(inp.b1, X, inp.W1))
            return a2(torch.addmm(inp.b2, H, inp.W2))
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / steps


def padded_rows(cfg, inp):
    """Rows of the grouped layout, zero padding included (each expert's rows
    rounded up to whole 256-row bands), from the routing the library returns."""
    _, r = moe_call(cfg, inp, inp.X, inp.logits, routing=True)
    counts = r["expert_offsets"].diff().cpu().tolist()
    return int(sum((c + 255) // 256 * 256 for c in counts))


def measure_gpu(name, args, world, rank, local, with_cpu):
    """One workload: device-timed steps, the dominant kernel's roofline, the
    end-to-end figures, clocks, and (rank 0, N = 1) the CPU oracle baseline.
    Returns the workload's entry of the JSON line."""
    import torch
    import transformer_ffn_gb300 as tffn

    cfg = CONFIGS[name]
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    inp = make_inputs(cfg, dev)
    out = torch.empty((cfg["M"], cfg["P"]), dtype=torch.bfloat16, device=dev)
    do_flush, l2_note = l2_policy(cfg, dev)
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if do_flush else None
    step = step_fn(cfg, inp, out)

    for _ in range(args.warmup):
        if flush_buf is not None:
            flush_buf.zero_()
        step()
    tffn.check()
    launches_per_step = tffn.last_launch_count()

    # ---- timed region (device time, inputs resident)
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    # one dominant-kernel launch in four gets its own event pair when the
    # steps run back to back (an event recorded between two kernels
    # serialises them and would slow every step it sits in)
    timing_every = 4 if flush_buf is None and args.steps >= 8 else 1
    tffn.timing_begin(timing_every)
    sampler.mark("start")
    t0 = time.perf_counter()
    per_step = time_steps(step, args.steps, flush_buf, stream)
    barrier(world)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    sampler.mark("end")
    n_dom, dom_ms = tffn.timing_end()
    clocks = sampler.stop()
    tffn.check()

    mean_s = sum(per_step) / len(per_step)
    mean_s = max_over_ranks(mean_s, world)
    metric, unit = metric_of(cfg)
    value = rate(cfg, mean_s) * world

    # ---- dominant kernel roofline (its own events, same steps)
    peak_tf, peak_gbs, peak_kind = measured_peaks()
    dom_s = dom_ms / 1e3 / max(n_dom, 1)
    if is_hbm_bound(cfg):
        roof = {"bound": "hbm", "achieved": weight_bytes(cfg) / dom_s / 1e9, "peak": peak_gbs,
                "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops(cfg) / dom_s / 1e12, "peak": peak_tf, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if not is_hbm_bound(cfg) and sustained_bf16_peak():
        # the burst peak is the denominator; a run of many steps meets the power cap
        # like the sustained measurement does, so that fraction is given for context
        roof["sustained_peak"] = sustained_bf16_peak()
        roof["frac_of_sustained"] = roof["achieved"] / roof["sustained_peak"]
    # the datasheet's dense peaks, for context (the fraction above is the one reported)
    roof["spec_peak"] = SPEC_HBM_GBS if is_hbm_bound(cfg) else SPEC_BF16_TFLOPS
    roof["frac_of_spec"] = roof["achieved"] / roof["spec_peak"]
    roof["peak_source"] = f"{peak_kind} (MEASURED_PEAKS.json {'hbm_gbs' if is_hbm_bound(cfg) else 'bf16_tflops'})"
    roof["kernel"] = dominant_kernel(name, args.ffn_path)
    roof["kernel_ms"] = dom_s * 1e3
    roof["kernel_launches_timed"] = n_dom
    roof["kernel_timing"] = (f"CUDA event pair around one launch of every {timing_every} in the timed region"
                             if timing_every > 1 else "CUDA event pair around every launch in the timed region")
    roof["algorithmic_per_launch"] = weight_bytes(cfg) if is_hbm_bound(cfg) else flops(cfg)
    roof["traffic"] = recorded_traffic(name, roof["kernel"])
    if weight_bytes(cfg) < 64e6 and is_hbm_bound(cfg):
        roof["note"] = ("launch/latency-bound: a step moves only "
                        f"{weight_bytes(cfg) / 1e6:.1f} MB, so its fraction of HBM is context, not a target")

    # ---- end to end through the public API.  Pipelined: every step uploads
    # its input from pinned host memory, runs the FFN and downloads its result,
    # step i+1's upload and step i-1's download overlapping step i's compute
    # (double-buffered device tensors, one stream per direction, ordered by
    # events).  Latency: the same, one call at a time with a synchronisation.
    e2e_mean, h2d, d2h = run_e2e(cfg, inp, args, flush_buf, stream)
    e2e_mean = max_over_ranks(e2e_mean, world)
    lat = run_e2e_latency(cfg, inp, args.steps, max(2, args.warmup), stream)
    lat_mean = max_over_ranks(sum(lat) / len(lat), world)

    entry = {
        "workload": cfg["label"], "metric": metric, "value": value, "unit": unit,
        "ms_per_step": mean_s * 1e3,
        "ms_per_step_min": min(per_step) * 1e3 if flush_buf is not None else None,
        "ms_per_step_std": statistics.pstdev(per_step) * 1e3 if flush_buf is not None else None,
        "timing": ("per-step event pairs, L2 flushed between steps" if flush_buf is not None
                   else "one event pair around the back-to-back steps"),
        "steps": args.steps,
        "l2": l2_note, "global_batch": cfg["M"] * world, "flops_per_step": flops(cfg),
        "roofline": roof,
        "e2e": {"value": rate(cfg, e2e_mean) * world, "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_mean * 1e3,
                "mode": "pipelined: upload of step i+1 and download of step i-1 overlap step i",
                "latency": {"value": rate(cfg, lat_mean) * world, "unit": unit, "ms_per_call": lat_mean * 1e3,
                            "ms_per_call_median": statistics.median(lat) * 1e3,
                            "mode": "one call at a time: upload, call, download, synchronise (host wall clock)"}},
        "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
        "wall_s_timed_block": wall,
    }
    if cfg["kind"] in ("ffn", "glu") and not args.no_unfused:
        u_s = max_over_ranks(run_unfused(cfg, inp, args.steps, max(2, args.warmup), stream), world)
        entry["unfused_comparator"] = {
            "impl": "the same FFN as separate kernels: cuBLAS GEMMs (torch.matmul / addmm) and torch "
                    "elementwise bias and activation kernels, H in bf16 between the layers",
            "value": rate(cfg, u_s) * world, "unit": unit, "ms_per_step": u_s * 1e3,
            "fused_speedup": u_s / mean_s}
    if args.ffn_path != "auto":
        entry["path"] = args.ffn_path
    if cfg["kind"] == "moe":
        entry["routed_rows"] = cfg["M"] * cfg["k"]
        entry["router"] = cfg.get("router", "balanced")
        entry["padded_rows"] = padded_rows(cfg, inp)
        entry["segment_order"] = "largest expert first" if args.moe_order else "expert index"
    if with_cpu and rank == 0 and world == 1 and not args.no_cpu_baseline:
        entry["cpu_baseline"] = cpu_baseline(name, cfg, inp, out.clone(), budget_s=args.cpu_budget)
    del inp, out, flush_buf
    torch.cuda.empty_cache()
    return entry


def _summary(entry):
    keep = ("workload", "metric", "value", "unit", "ms_per_step")
    s = {k: entry[k] for k in keep}
    s["frac"] = entry["roofline"]["frac"]
    s["kernel_ms"] = entry["roofline"]["kernel_ms"]
    s["kernel_achieved"] = entry["roofline"]["achieved"]
    s["e2e_latency_ms"] = entry["e2e"]["latency"]["ms_per_call"]
    if "unfused_comparator" in entry:
        s["fused_speedup_vs_unfused"] = entry["unfused_comparator"]["fused_speedup"]
    return s


def run_gpu(args, world, rank, local):
    import transformer_ffn_gb300 as tffn

    tffn.load()
    tffn.set_option(tffn.OPT_MOE_ORDER, args.moe_order)
    tffn.set_option(tffn.OPT_PATH, FFN_PATHS[args.ffn_path])
    names = list(SUITE) if args.config == "all" else [args.config]
    head = HEADLINE if args.config == "all" else args.config
    entries = {n: measure_gpu(n, args, world, rank, local, with_cpu=True) for n in names}
    e = entries[head]
    line = {
        "metric": e["metric"], "value": e["value"], "unit": e["unit"], "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": e["ms_per_step"], "ms_per_step_min": e["ms_per_step_min"],
        "ms_per_step_std": e["ms_per_step_std"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; X~N(0,1), W~N(0,1/fan_in), b~U(-0.1,0.1), bf16)",
        "config": {"workload": e["workload"], "parallelism": f"replicas{world}" if world > 1 else "single GPU",
                   "l2": e["l2"], "timing": e["timing"], "global_batch": e["global_batch"],
                   "flops_per_step": e["flops_per_step"]},
        "roofline": e["roofline"], "e2e": e["e2e"], "clocks": e["clocks"], "gpu_launches": e["gpu_launches"],
        "wall_s_timed_block": e["wall_s_timed_block"],
    }
    for k in ("path", "routed_rows", "router", "padded_rows", "segment_order"):
        if k in e:
            line["config"][k] = e[k]
    if "cpu_baseline" in e:
        line["cpu_baseline"] = e["cpu_baseline"]
    if len(entries) > 1:
        line["config"]["headline"] = head
        line["configs"] = entries
        # the metric's two halves side by side: weight GB/s at small M (the
        # decode workload), TFLOP/s at the largest M (the large workload)
        if "decode" in entries:
            line["small_m"] = _summary(entries["decode"])
        if "large" in entries:
            line["large_m"] = _summary(entries["large"])
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------- oracle (CPU) arms
def _oracle_inputs(cfg, inp):
    from transformer_ffn_gb300 import synth
    u = synth.to_u16
    if cfg["kind"] == "glu":
        return (u(inp.X), u(inp.W1), u(inp.W3), u(inp.W2))
    if cfg["kind"] == "moe" and cfg.get("glu"):
        return (u(inp.X), inp.logits.cpu().numpy(), [u(w) for w in inp.W1], [u(w) for w in inp.W3],
                [u(w) for w in inp.W2])
    if cfg["kind"] == "moe":
        return (u(inp.X), inp.logits.cpu().numpy(), [u(w) for w in inp.W1], [u(b) for b in inp.b1],
                [u(w) for w in inp.W2], [u(b) for b in inp.b2])
    return (u(inp.X), u(inp.W1), u(inp.b1), u(inp.W2), u(inp.b2))


def _oracle_rows(cfg, host, rows):
    import oracle
    acts = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu_tanh": oracle.ACT_GELU_TANH,
            "silu": oracle.ACT_SILU}
    if cfg["kind"] == "glu":
        X, W1, W3, W2 = host
        return oracle.glu_ffn(X, W1, W3, W2, acts[cfg["act1"]], rows=rows)
    if cfg["kind"] == "moe" and cfg.get("glu"):
        X, lg, W1, W3, W2 = host
        return oracle.moe_glu_ffn(X, lg, cfg["k"], W1, W3, W2, acts[cfg["act1"]], tokens=rows)
    if cfg["kind"] == "moe":
        X, lg, W1, b1, W2, b2 = host
        return oracle.moe_ffn(X, lg, cfg["k"], W1, b1, W2, b2, acts[cfg["act1"]], acts[cfg["act2"]],
                              tokens=rows)
    X, W1, b1, W2, b2 = host
    return oracle.ffn(X, W1, b1, W2, b2, acts[cfg["act1"]], acts[cfg["act2"]], rows=rows)


def _sample_work(cfg, nrows):
    """Algorithmic work of nrows of the workload, in the metric's unit base."""
    if is_hbm_bound(cfg):
        return weight_bytes(cfg) * nrows / cfg["M"]     # share of the step's bytes
    return flops(cfg) * nrows / cfg["M"]


def host_cpu():
    """The host CPU's model name and logical core count."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        import platform
        model = platform.processor() or platform.machine()
    return {"model": model, "cores": os.cpu_count()}


# Workloads the oracle runs in full (a few seconds of fp64 work); the others
# are sampled (random rows until the time budget) and their full-workload
# time is extrapolated linearly from the sample.
CPU_FULL = ("tiny", "decode")


def cpu_baseline(name, cfg, inp, Y_dev=None, budget_s=8.0):
    """The oracle, as it stands, single-threaded on rows of the same workload:
    every row for the workloads in CPU_FULL, else one random row at a time
    until about budget_s seconds of work."""
    import numpy as np
    host = _oracle_inputs(cfg, inp)
    full = name in CPU_FULL
    rng = np.random.default_rng(0)
    order = list(range(cfg["M"])) if full else rng.permutation(cfg["M"])
    done, t_total = [], 0.0
    results = []
    if full:
        t0 = time.perf_counter()
        results = list(_oracle_rows(cfg, host, order))
        t_total = time.perf_counter() - t0
        done = order
    else:
        while t_total < budget_s and len(done) < cfg["M"]:
            r = int(order[len(done)])
            t0 = time.perf_counter()
            y = _oracle_rows(cfg, host, [r])
            t_total += time.perf_counter() - t0
            done.append(r)
            results.append(y[0])
    metric, unit = metric_of(cfg)
    what = "tokens" if cfg["kind"] == "moe" else "rows"
    out = {"value": (_sample_work(cfg, len(done)) / t_total) / (1e9 if unit == "GB/s" else 1e12),
           "unit": unit, "cores": 1, "kind": "oracle",
           "sample": (f"all {cfg['M']} {what}" if full else f"{len(done)} random of {cfg['M']} {what}") +
                     f" ({cfg['label']}), single-threaded C oracle, fp64 accumulation",
           "seconds": t_total, "host": host_cpu()}
    if full:
        out["full_workload_s"] = t_total
    else:
        out["extrapolated"] = True
        out["full_workload_s_extrapolated"] = t_total * cfg["M"] / len(done)
    # the same rows, row-parallel over every host core (ctypes releases the
    # interpreter lock during each C call): a second figure, labelled as such
    from concurrent.futures import ThreadPoolExecutor
    nthr = max(1, min(os.cpu_count() or 1, len(done)))
    rows = [int(r) for r in done]
    chunks = [rows[i * len(rows) // nthr:(i + 1) * len(rows) // nthr] for i in range(nthr)]
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=nthr) as ex:
        list(ex.map(lambda c: _oracle_rows(cfg, host, c), [c for c in chunks if c]))
    t_all = time.perf_counter() - t0
    out["all_cores"] = {"value": (_sample_work(cfg, len(done)) / t_all) / (1e9 if unit == "GB/s" else 1e12),
                        "unit": unit, "cores": nthr, "seconds": t_all,
                        "kind": "oracle, the same rows split over host threads (row-parallel)"}
    if Y_dev is not None:
        got = Y_dev[list(done)].float().cpu().numpy()
        want = np.stack(results)
        err = np.abs(got - want)
        out["parity_on_sample"] = bool(np.all(err <= 1e-2 + 1e-2 * np.abs(want)))
        out["max_abs_err_on_sample"] = float(err.max())
    return out


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle timed on host cores, same metric."""
    if rank != 0:
        return
    name = HEADLINE if args.config == "all" else args.config
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, "cpu")
    import numpy as np
    host = _oracle_inputs(cfg, inp)
    rows_per_step = max(1, int(args.ref_rows))
    rng = np.random.default_rng(1)
    for _ in range(args.warmup):
        _oracle_rows(cfg, host, [int(x) for x in rng.choice(cfg["M"], size=1)])
    times = []
    for _ in range(args.steps):
        rows = [int(x) for x in rng.choice(cfg["M"], size=rows_per_step, replace=False)]
        t0 = time.perf_counter()
        _oracle_rows(cfg, host, rows)
        times.append(time.perf_counter() - t0)
    mean_s = sum(times) / len(times)
    metric, unit = metric_of(cfg)
    val = (_sample_work(cfg, rows_per_step) / mean_s) / (1e9 if unit == "GB/s" else 1e12)
    sample = (f"{rows_per_step} random rows of {cfg['M']} per step ({cfg['label']}), "
              f"single-threaded C oracle, fp64 accumulation")
    line = {"impl": "reference", "metric": metric, "value": val, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_s * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, same recipe as the GPU arm)",
            "config": {"workload": cfg["label"], "rows_per_step": rows_per_step},
            "cpu_baseline": {"value": val, "unit": unit, "cores": 1, "kind": "oracle", "sample": sample,
                             "host": host_cpu()},
            "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 200 on the GPU, whose steps take 0.05-10 ms, so that the "
                         "clock samples fall inside the timed region; 20 for the CPU reference arm)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT, choices=sorted(CONFIGS) + ["all"],
                    help="workload; 'all' (default) measures " + ", ".join(SUITE) + " with " + HEADLINE +
                         " as the headline")
    ap.add_argument("--ffn-path", default="auto", choices=sorted(FFN_PATHS),
                    help="dense FFN path: auto, fused (engine), decode, two (two launches), "
                         "reduce (the reduce-add form of the fused-FFN page, section Step 1), "
                         "b2b (back-to-back, H on chip), stream (tensor-core weight stream)")
    ap.add_argument("--moe-order", type=int, default=1, choices=(0, 1),
                    help="MoE grouped-layout segment order: 0 expert index, 1 largest expert first")
    ap.add_argument("--impl", default="tffn", choices=["tffn", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=8.0,
                    help="seconds of oracle work per sampled workload in the CPU baseline")
    ap.add_argument("--ref-rows", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-unfused", action="store_true",
                    help="skip the unfused comparator (cuBLAS GEMMs + torch elementwise kernels)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 20 if args.impl == "reference" else 200
    if args.warmup < 3 and args.impl != "reference":
        args.warmup = 3
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_gpu(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
