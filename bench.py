#!/usr/bin/env python
"""Decode throughput of the fp32 Llama-2 decode library on B300.

One step = one greedy generation of the named workload (every forward of its
prompt and generated positions) through the library's C ABI. Default workload:
the 7B shape at batch 1 (64-token prompt + 256 generated tokens = 319
forwards), the largest configuration that fits one GPU; the default line also
carries a "batch256" object, the batched workload (256 sequences on the 44M
shape, prompts of 1-128 tokens, 512 generated tokens each) measured the same
way.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 7b|15m|44m|110m|batched]
    python bench.py --impl reference ...   # the C oracle on the host cores
    python bench.py --kernel-only 3 --layers 2   # one kernel kind on a reduced-depth
                                                 # model of the same shape (ncu case)

Prints ONE JSON line (rank 0). N > 1 runs under torchrun: every rank decodes
its own replica (batch-1 decode does not shard; no collective on the data
path), `value` is the sum over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "decode tok/s (fp32, batch 1)"
METRIC_BATCHED = "decode tok/s (fp32, batch 256)"
DOMINANT_KIND = 3  # W1/W3 + SwiGLU: 44% of the streamed bytes of a 7B-shape step
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "w13_swiglu_7b_shape.md")
KERNEL_SOURCE = os.path.join(ROOT, "llama_fp32_token_decode_b300", "csrc", "matvec.cu")
BATTN_PROFILE = os.path.join(ROOT, "profiles", "battn_batched_44m.md")
BATTN_SOURCE = os.path.join(ROOT, "llama_fp32_token_decode_b300", "csrc", "batched.cu")
BATTN_HEAD = "template <int LPR, int G, int MINB>\n__global__ void"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="7b", choices=["15m", "44m", "110m", "7b", "batched"])
    ap.add_argument("--no-prefill", action="store_true",
                    help="7B run: skip the with-prefill measurement (and its tf32 weight copies)")
    ap.add_argument("--no-batched", action="store_true",
                    help="default run: skip the batch-256 measurement added to the 7B line")
    ap.add_argument("--cpu-forwards", type=int, default=0,
                    help="oracle forwards in the CPU-baseline sample (0 = about 20 s worth)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-small", action="store_true",
                    help="default run: skip the 15m / 44m / 110m batch-1 lines")
    ap.add_argument("--kernel-only", type=int, default=None,
                    help="time one kernel kind (0 QKV, 1 attention, 2 Wo, 3 W1/W3, 4 W2, "
                         "5 classifier; 6-13 the batched kinds with --workload batched "
                         "(8-10 with --workload 7b: the prefill pass's GEMMs on its 64 rows); "
                         "14 attention block, 15 FFN block on a two-kernels-per-layer "
                         "workload: 15m, 44m, 110m) on the workload's shape and exit: the "
                         "profiling case")
    ap.add_argument("--layers", type=int, default=0,
                    help="with --kernel-only: layers of the reduced-depth model (0 = all)")
    return ap.parse_args()


# ---------------------------------------------------------------- helpers

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


REJECT_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(clocks) -> bool:
    """A timed region is not a valid measurement when the GPU slowed down
    (hardware or thermal reason), or when the SM clock sat well below its
    maximum with no reason at all (a clock lock left by someone else)."""
    if not clocks:
        return False
    if any(r in REJECT_REASONS for r in clocks["reasons"]):
        return True
    return (not clocks["reasons"] and clocks["sm_max_mhz"] > 0
            and clocks["sm_mhz"] < 0.8 * clocks["sm_max_mhz"])


def timed_steps(step, stream, steps, world, local):
    """K steps between CUDA events on `stream`, barrier + synchronize on both
    sides, clocks sampled meanwhile; max over ranks. A region whose clocks are
    rejected (on any rank) is measured once more and the second one is
    reported. Returns (ms, clocks, remeasured)."""
    import torch
    for attempt in range(2):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.3)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize()
        clocks = sampler.stop()
        barrier(world)
        ms_max = max_over_ranks(e0.elapsed_time(e1), world)
        bad = max_over_ranks(1.0 if clocks_rejected(clocks) else 0.0, world) > 0
        if not bad or attempt == 1:
            if clocks is not None:
                clocks["remeasured"] = attempt == 1
            return ms_max, clocks, attempt == 1


def forwards_of(w) -> int:
    return w["n_prompt"] + w["steps"] - 1


def workload_bytes_per_forward(cfg, pos: float) -> float:
    """Algorithmic HBM bytes of one batch-1 forward at position pos: every weight
    except the embedding table, one embedding row, and the KV rows read and
    written."""
    d, F, L, V = cfg["dim"], cfg["hidden_dim"], cfg["n_layers"], cfg["vocab_size"]
    kvd = cfg["n_kv_heads"] * (d // cfg["n_heads"])
    weights = L * (2 * d * d + 2 * d * kvd + 3 * d * F + 2 * d) + d + V * d
    kv = L * (2 * kvd * (pos + 1) + 2 * kvd)
    return 4.0 * (weights + d + kv)


def batched_run_bound(cfg, lens, steps: int, B: int, hbm_gbs: float, p3_tflops: float):
    """Lower bound (seconds) of one batched generation run, phase by phase.

    Lockstep step t runs every sequence at position t; sequence b is active
    for t < lens[b] + steps - 1 (inactive rows stay in the GEMMs). A step's
    GEMM phase cannot beat max(its fp32 weights once / HBM, its FLOPs on all
    B rows / 3xTF32 peak); its attention phase cannot beat the KV bytes of the
    active rows (read positions 0..t, write position t) / HBM. The phases are
    dependent, so their bounds add; the embedding rows and norm vectors are
    counted with the weights."""
    d, F, L, V = cfg["dim"], cfg["hidden_dim"], cfg["n_layers"], cfg["vocab_size"]
    kvd = cfg["n_kv_heads"] * (d // cfg["n_heads"])
    weights = 4.0 * (L * (2 * d * d + 2 * d * kvd + 3 * d * F + 2 * d) + d + V * d + B * d)
    flops = 2.0 * B * (L * (d * (d + 2 * kvd) + d * d + 3 * d * F) + V * d)
    gemm_s = max(weights / (hbm_gbs * 1e9), flops / (p3_tflops * 1e12))
    n_lock = int(lens.max()) + steps - 1
    t = np.arange(n_lock)
    active = (t[:, None] < (lens[None, :] + steps - 1)).sum(axis=1)
    kv_bytes = 4.0 * L * 2 * kvd * active * (t + 2)  # read t + 1 rows, write 1
    return n_lock * gemm_s + float(kv_bytes.sum()) / (hbm_gbs * 1e9), n_lock * gemm_s


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_median": statistics.median(power) if power else None}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6400.0}, "fallback"


_FP32_PEAKS = None


def measured_fp32_peaks():
    """Dense fp32-input GEMM peaks measured live on this GPU with the library
    GEMM (cuBLAS through torch.matmul, 8192^3, best of 5 after warm-up): TF32
    tensor cores (allow_tf32) and plain SGEMM (FFMA). None when not measurable."""
    global _FP32_PEAKS
    if _FP32_PEAKS is not None:
        return _FP32_PEAKS
    try:
        import torch
        n = 8192
        g = torch.Generator(device="cuda").manual_seed(0)
        a = torch.randn(n, n, device="cuda", generator=g)
        b = torch.randn(n, n, device="cuda", generator=g)
        out = {}
        old = torch.backends.cuda.matmul.allow_tf32
        for name, tf in (("tf32_tflops", True), ("sgemm_tflops", False)):
            torch.backends.cuda.matmul.allow_tf32 = tf
            for _ in range(2):
                a @ b
            best = float("inf")
            for _ in range(5):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                a @ b
                e1.record()
                e1.synchronize()
                best = min(best, e0.elapsed_time(e1))
            out[name] = 2.0 * n ** 3 / (best / 1e3) / 1e12
        torch.backends.cuda.matmul.allow_tf32 = old
        del a, b
        torch.cuda.empty_cache()
        _FP32_PEAKS = out
    except Exception:  # noqa: BLE001  (a probe failure only changes the denominator's source)
        _FP32_PEAKS = {}
    return _FP32_PEAKS


def tf32x3_peak(peaks):
    """Peak of the 3xTF32 GEMM in fp32-equivalent TFLOP/s and its source: the
    TF32 tensor peak measured live (cuBLAS TF32, burst) divided by the three
    tensor passes per product; without it, the measured bf16 dense peak times
    the nominal tf32/bf16 ratio (1.1 / 2.25 PFLOP/s), divided by three."""
    m = measured_fp32_peaks()
    if m.get("tf32_tflops"):
        return m["tf32_tflops"] / 3.0, "measured live: cuBLAS TF32 8192^3 (burst) / 3"
    bf16 = float(peaks.get("bf16_tflops", 1800.0))
    return bf16 * (1.1 / 2.25) / 3.0, "measured bf16_tflops x 1.1/2.25 / 3 (nominal ratio)"


def summary_values(path):
    """The `- key: value` lines of a committed ncu summary, or None."""
    try:
        txt = open(path).read()
    except OSError:
        return None
    vals = {}
    for ln in txt.splitlines():
        if ":" in ln and ln.strip().startswith("- "):
            k, v = ln.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    return vals


def kernel_text_sha256(path, head):
    """sha256 of one kernel's source text: from the line that starts with
    `head` to the first closing brace in column 0 after it (None if absent)."""
    src = open(path).read()
    i = src.find(head)
    if i < 0:
        return None
    j = src.find("\n}\n", i)
    if j < 0:
        return None
    return hashlib.sha256(src[i:j + 3].encode()).hexdigest()


def profiled_traffic():
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu summary,
    or None when the summary is missing or the kernel source changed since."""
    vals = summary_values(PROFILE_TRAFFIC)
    if vals is None:
        return None
    src = hashlib.sha256(open(KERNEL_SOURCE, "rb").read()).hexdigest()
    if vals.get("matvec.cu sha256") != src:
        return None
    try:
        return float(vals["dram bytes per 7B-shape launch (read + write)"])
    except (KeyError, ValueError):
        return None


def profiled_battn_traffic(alg_bytes):
    """Per-launch DRAM bytes of the batched attention at the timed position:
    the captured launch's DRAM bytes over its algorithmic bytes (K and V rows
    read once per position, so both grow with the positions) times this
    launch's algorithmic bytes. None when the summary is missing or the
    kernel's source text changed since the capture."""
    vals = summary_values(BATTN_PROFILE)
    if vals is None or vals.get("battn4_kernel source sha256") != kernel_text_sha256(
            BATTN_SOURCE, BATTN_HEAD):
        return None
    try:
        dram = float(vals["dram bytes per launch (read + write)"])
        alg = float(vals["algorithmic bytes per launch"])
    except (KeyError, ValueError):
        return None
    return dram / alg * alg_bytes


def oracle_sample(cfg, blob, prompt, n_fwd: int):
    """Times the oracle, as it stands, over the first n_fwd forwards."""
    import oracle
    m = oracle.Model(cfg, blob)
    tok = int(prompt[0])
    t0 = time.perf_counter()
    for p in range(n_fwd):
        lg = m.forward(tok, p)
        tok = int(prompt[p + 1]) if p + 1 < len(prompt) else int(np.argmax(lg))
    dt = time.perf_counter() - t0
    m.close()
    return dt


def default_cpu_forwards(name: str) -> int:
    # about 10-25 s of one core per sample
    # (7b: the first 8 forwards, the sample its configuration fixes: about a minute)
    return {"15m": 256, "44m": 120, "110m": 40, "7b": 8, "batched": 120}[name]


# ---------------------------------------------------------------- reference arm

def run_reference(args, world, rank):
    if rank != 0:
        return 0
    w = synth.workload(args.workload)
    cfg = synth.model_config(w)
    blob = synth.make_blob(cfg, w["seed"])
    if w["prompt"] == "batch":  # sequences are independent: time sequence 0
        lens, prompts = synth.batch_inputs(w)
        prompt = prompts[:lens[0]]
    else:
        prompt = synth.prompt(w)
    if args.workload == "7b":
        # one forward per step over the first 8 positions, in order and then
        # again (the cache keeps the earlier positions): the configuration times
        # the oracle on its first 8 steps, a step of seconds each
        import oracle
        per_step = 1
        m = oracle.Model(cfg, blob)
        toks = [int(t) for t in prompt[:8]]
        k = 0

        def one():
            nonlocal k
            p = k % 8
            t0 = time.perf_counter()
            m.forward(toks[p], p)
            k += 1
            return time.perf_counter() - t0

        for _ in range(args.warmup):
            one()
        t = sum(one() for _ in range(args.steps))
        m.close()
        sample = ("one forward per step, positions 0..7 of the 7b workload's prompt in turn "
                  "(its first 8 steps), single-threaded C oracle (-O2, no fast-math)")
    else:
        per_step = max(1, (args.cpu_forwards or default_cpu_forwards(args.workload)) // 2)
        for _ in range(args.warmup):
            oracle_sample(cfg, blob, prompt, 1)
        t = sum(oracle_sample(cfg, blob, prompt, per_step) for _ in range(args.steps))
        sample = (f"first {per_step} forwards (positions 0..{per_step - 1}) of the "
                  f"{args.workload} workload per step, single-threaded C oracle (-O2, no "
                  f"fast-math)")
    value = args.steps * per_step / t
    line = {"impl": "reference",
            "metric": METRIC_BATCHED if args.workload == "batched" else METRIC, "value": value, "unit": "tok/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": args.workload, "global_batch": 1,
                       "dim": cfg["dim"], "n_layers": cfg["n_layers"], "n_heads": cfg["n_heads"],
                       "n_kv_heads": cfg["n_kv_heads"], "hidden_dim": cfg["hidden_dim"],
                       "vocab_size": cfg["vocab_size"], "seq_len": cfg["seq_len"],
                       "forwards_per_step": per_step, "parallelism": "replicas1",
                       "sample_of": ("sequence 0 of the 256-sequence batched workload"
                                     if w["prompt"] == "batch" else
                                     f"the {args.workload} generation")},
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm

def upload_blob_in_pieces(cfg, seed):
    """The seeded blob drawn in 256 MB pieces straight into a device tensor, so
    that no rank holds the whole blob in host memory."""
    import torch
    n = synth.blob_floats(cfg)
    d_blob = torch.empty(n, dtype=torch.float32, device="cuda")
    chunk = 1 << 26
    host = torch.empty(chunk, dtype=torch.float32).pin_memory()
    h = host.numpy()
    off = 0
    for _, cnt, is_gain in synth.blob_segments(cfg):
        done = 0
        while done < cnt:
            m = min(chunk, cnt - done)
            if is_gain:
                h[:m] = 1.0
            else:
                synth._lib().synth_fill_normal(seed, synth.STREAM_WEIGHTS, off + done, m,
                                               synth.WEIGHT_STD, h.ctypes.data,
                                               os.cpu_count() or 1)
            d_blob[off + done:off + done + m].copy_(host[:m])
            done += m
        off += cnt
    torch.cuda.synchronize()
    return d_blob


def run_ours(args, world, rank, local):
    import torch

    import llama_fp32_token_decode_b300 as l2

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    w = synth.workload(args.workload)
    cfg = synth.model_config(w)
    use_prefill = args.workload == "7b" and not args.no_prefill
    if use_prefill:
        cfg["max_prefill"] = w["n_prompt"]  # rows of the prefill pass (no extra KV caches)
    n_fwd = forwards_of(w)
    prompt = synth.prompt(w)
    steps = w["steps"]
    keep_host_blob = (rank == 0 and world == 1 and not args.no_cpu_baseline)

    if keep_host_blob:  # the CPU baseline needs the blob on the host
        blob = synth.make_blob(cfg, w["seed"])
        dec = l2.Decoder(cfg, blob)
    else:
        blob = None
        d_blob = upload_blob_in_pieces(cfg, w["seed"])
        dec = l2.Decoder(cfg, d_blob=d_blob)
        del d_blob
        torch.cuda.empty_cache()

    stream = torch.cuda.Stream()
    d_prompt = torch.tensor(prompt, dtype=torch.int32, device="cuda")
    d_out = torch.zeros(steps, dtype=torch.int32, device="cuda")

    def step():
        l2.l2_generate_device(dec.h, d_prompt, len(prompt), steps, d_out, stream)

    for _ in range(args.warmup):
        step()
    stream.synchronize()
    ref_tokens = d_out.cpu().numpy().copy()

    # ---- timed region: K generations, inputs resident in HBM
    ms_max, clocks, _ = timed_steps(step, stream, args.steps, world, local)
    value = world * args.steps * n_fwd / (ms_max / 1e3)
    assert np.array_equal(d_out.cpu().numpy(), ref_tokens), "generation is not reproducible"

    # ---- end to end through the public host API: pinned host prompt in, tokens out
    h_prompt = torch.tensor(prompt, dtype=torch.int32).pin_memory().numpy()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        toks = dec.generate(h_prompt, steps)
    t_e2e = time.perf_counter() - t0
    t_e2e = max_over_ranks(t_e2e, world)
    assert np.array_equal(toks, ref_tokens), "host and device entry points disagree"
    e2e = {"value": world * args.steps * n_fwd / t_e2e, "unit": "tok/s",
           "h2d_bytes_per_step": int(h_prompt.nbytes), "d2h_bytes_per_step": int(steps * 4)}

    # ---- roofline of the dominant kernel, timed live on the launching stream
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    pos_mid = n_fwd // 2
    iters = 3 * cfg["n_layers"]
    k_ms = l2.l2_time_kernel(dec.h, DOMINANT_KIND, pos_mid, iters, stream)
    k_bytes = l2.l2_kernel_bytes(dec.h, DOMINANT_KIND, pos_mid)
    achieved = k_bytes / (k_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak,
                "traffic": profiled_traffic() if args.workload == "7b" else None,
                "kernel": "matvec_kernel<EPI_SWIGLU> (W1/W3 + SwiGLU)",
                "algorithmic_bytes_per_launch": k_bytes, "launch_ms": k_ms,
                "peak_source": f"{peak_kind} hbm_gbs (copy, burst)"}
    # every kernel kind of the forward, timed live at the same position
    kinds = {}
    for kind in range(6):
        t = median_time(l2, dec.h, kind, pos_mid, iters if kind < 5 else 8, stream)
        b = l2.l2_kernel_bytes(dec.h, kind, pos_mid)
        kinds[l2.KERNEL_KINDS[kind]] = {
            "launch_ms": t, "GB/s": b / (t / 1e3) / 1e9, "frac": b / (t / 1e3) / 1e9 / peak,
            "ms_per_forward": t * (cfg["n_layers"] if kind < 5 else 1)}
    roofline["per_kernel_at_pos"] = {"pos": pos_mid, "kernels": kinds}
    # whole-step roofline: algorithmic bytes of every forward over the step time
    step_bytes = sum(workload_bytes_per_forward(cfg, p) for p in range(n_fwd))
    step_gbs = step_bytes * args.steps / (ms_max / 1e3) / 1e9
    step_roofline = {"achieved": step_gbs, "peak": peak, "unit": "GB/s", "frac": step_gbs / peak,
                     "bytes_per_step": step_bytes,
                     "roofline_tok_s": n_fwd / (step_bytes / (peak * 1e9))}

    # ---- CPU baseline: the oracle as it stands, on a bounded sample, 1 core
    # ---- the same workload with the prompt taken by one prefill pass: the
    # decode of the generated tokens is unchanged, the 64 prompt positions go
    # through the tensor-core path at once (weights read once for the prompt)
    prefill = None
    if use_prefill:
        d_out_p = torch.zeros(steps, dtype=torch.int32, device="cuda")

        def pstep(k):
            l2.l2_generate_prefill_device(dec.h, d_prompt, len(prompt), k, d_out_p, stream)

        for _ in range(args.warmup):
            pstep(steps)
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            pstep(steps)
        e1.record(stream)
        e1.synchronize()
        ms_p = e0.elapsed_time(e1) / args.steps
        ptoks = d_out_p.cpu().numpy()
        same = int(np.argmax(ptoks != ref_tokens)) if np.any(ptoks != ref_tokens) else steps
        e0.record(stream)
        for _ in range(args.steps):
            pstep(1)  # the prefill pass alone (+ the hand-off of its argmax)
        e1.record(stream)
        e1.synchronize()
        ms_pre = e0.elapsed_time(e1) / args.steps
        d, F, L, V = cfg["dim"], cfg["hidden_dim"], cfg["n_layers"], cfg["vocab_size"]
        kvd = cfg["n_kv_heads"] * (d // cfg["n_heads"])
        params = L * (2 * d * d + 2 * d * kvd + 3 * d * F) + V * d
        n = len(prompt)
        flops = 2.0 * n * params
        bytes_fp32 = 4.0 * params
        peaks, _ = measured_peaks()
        p3, _ = tf32x3_peak(peaks)
        bound_ms = max(bytes_fp32 / (float(peaks["hbm_gbs"]) * 1e6), flops / (p3 * 1e9))
        prefill = {"value": n_fwd / (ms_p / 1e3), "unit": "tok/s", "ms_per_step": ms_p,
                   "prefill_ms": ms_pre, "prefill_tok_s": n / (ms_pre / 1e3),
                   "prefill_roofline": {
                       "bound_ms": bound_ms, "frac": bound_ms / ms_pre,
                       "flops": flops, "fp32_weight_bytes": bytes_fp32,
                       "note": "bound = max(fp32 weights once / HBM peak, 2 n params FLOPs / "
                               "3xTF32 peak); the pass reads each weight once in fp32 "
                               "(times its folded RMSNorm gain) and splits it into the "
                               "tf32 pair in shared memory"},
                   "tokens_equal_to_decode_path": same,
                   "note": "prompt through l2_generate_prefill_device (one causal "
                           "tensor-core pass), then 255 decode forwards; not the headline"}

    cpu = None
    if keep_host_blob:
        nf = args.cpu_forwards or default_cpu_forwards(args.workload)
        dt = oracle_sample(cfg, blob, prompt, nf)
        cpu = {"value": nf / dt, "unit": "tok/s", "cores": 1, "kind": "oracle",
               "sample": f"first {nf} forwards (positions 0..{nf - 1}) of the {args.workload} "
                         f"workload, single-threaded C oracle (-O2, no fast-math), "
                         f"host has {os.cpu_count()} cores"}

    launches_per_step = n_fwd * (5 * cfg["n_layers"] + 1) + 1
    line = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (random-init N(0,0.02) weights, seeded prompt ids)",
            "config": {"workload": args.workload, "global_batch": world,
                       "dim": cfg["dim"], "n_layers": cfg["n_layers"], "n_heads": cfg["n_heads"],
                       "hidden_dim": cfg["hidden_dim"], "vocab_size": cfg["vocab_size"],
                       "seq_len": cfg["seq_len"], "n_prompt": w["n_prompt"],
                       "generated": steps, "forwards_per_step": n_fwd,
                       "parallelism": f"replicas{world}",
                       "l2": "inputs larger than L2 (%.2f GB streamed per forward)" % (
                           step_bytes / n_fwd / 1e9) if step_bytes / n_fwd > 126e6 else
                       "weights may stay L2-resident (%.1f MB per forward)" % (
                           step_bytes / n_fwd / 1e6)},
            "roofline": roofline, "step_roofline": step_roofline,
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": launches_per_step * args.steps}
    if prefill is not None:
        line["with_prefill"] = prefill
    dec.close()
    del dec
    if blob is not None:
        del blob
    torch.cuda.empty_cache()
    if args.workload == "7b" and not args.no_small:
        line["small_models"] = run_small_models(args, world, local)
    if args.workload == "7b" and not args.no_batched:
        # the other half of the metric: batch 256 on the 44M shape, same process
        line["batch256"] = run_ours_batched(args, world, rank, local, compact=True)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_small_models(args, world, local):
    """The pages' small shapes at batch 1 (15m: dim 288 / 6 layers; 44m: dim 512
    / 8 layers, context 1024; 110m: dim 768 / 12 layers), each a full greedy
    generation per step through l2_generate_device, timed like the headline.
    Their weights (62 / 184 / 476 MB per forward) sit partly or wholly in the
    126 MB L2, so a forward is bound by the latency of its dependent kernels
    rather than by HBM; the HBM fraction is reported all the same."""
    import torch

    import llama_fp32_token_decode_b300 as l2
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    out = {}
    for name in ("15m", "44m", "110m"):
        w = synth.workload(name)
        cfg = synth.model_config(w)
        prompt = synth.prompt(w)
        steps, n_fwd = w["steps"], forwards_of(w)
        blob = synth.make_blob(cfg, w["seed"])
        with l2.Decoder(cfg, blob) as dec:
            del blob
            layer_kernels = l2.l2_layer_kernels(dec.h)
            stream = torch.cuda.Stream()
            d_prompt = torch.tensor(prompt, dtype=torch.int32, device="cuda")
            d_out = torch.zeros(steps, dtype=torch.int32, device="cuda")

            def step():
                l2.l2_generate_device(dec.h, d_prompt, len(prompt), steps, d_out, stream)

            for _ in range(args.warmup):
                step()
            stream.synchronize()
            ms_max, clocks, _ = timed_steps(step, stream, args.steps, world, local)
        step_bytes = sum(workload_bytes_per_forward(cfg, p) for p in range(n_fwd))
        tok_s = world * args.steps * n_fwd / (ms_max / 1e3)
        gbs = step_bytes * args.steps / (ms_max / 1e3) / 1e9
        out[name] = {"value": tok_s, "unit": "tok/s", "ms_per_step": ms_max / args.steps,
                     "forwards_per_step": n_fwd, "us_per_forward": ms_max * 1e3 / args.steps / n_fwd,
                     "step_roofline": {"achieved": gbs, "peak": hbm, "unit": "GB/s",
                                       "frac": gbs / hbm,
                                       "bytes_per_forward": step_bytes / n_fwd,
                                       "peak_source": f"{peak_kind} hbm_gbs (copy, burst)"},
                     # weights under 100 MB are kept in L2 (evict_last) from
                     # token to token: their bytes then come from L2, not HBM
                     "weights_in_l2": bool(step_bytes / n_fwd < 100e6),
                     "layer_kernels": layer_kernels,
                     "kernels_per_forward": layer_kernels * cfg["n_layers"] + 1,
                     "clocks": clocks}
    return out


BATCHED_KINDS = {  # batched kernel kinds of l2_time_kernel and their launches per step
    6: "QKV GEMM (+RoPE, KV append)", 7: "attention", 8: "Wo GEMM (+residual)",
    9: "W1/W3 GEMM (+SwiGLU)", 10: "W2 GEMM (+residual)", 11: "classifier GEMM (+argmax)",
    12: "embedding gather"}


def batched_gemm_shape(cfg, kind):
    """(N, K) of a batched GEMM kind, or None for the non-GEMM kinds."""
    d, F, V = cfg["dim"], cfg["hidden_dim"], cfg["vocab_size"]
    kvd = cfg["n_kv_heads"] * (d // cfg["n_heads"])
    return {6: (d + 2 * kvd, d), 8: (d, d), 9: (2 * F, d), 10: (d, F), 11: (V, d)}.get(kind)


def median_time(l2, h, kind, pos, iters, stream, reps=3):
    """Per-launch time of one kernel kind: the median of `reps` timed loops of
    `iters` launches (one loop can catch a clock or scheduling excursion)."""
    return float(np.median([l2.l2_time_kernel(h, kind, pos, iters, stream) for _ in range(reps)]))


def run_ours_batched(args, world, rank, local, compact=False):
    """Batch 256 on the 44M shape: one step = one l2_generate_batch_device of
    the whole workload (every sequence's prompt and generated positions,
    lockstep), tokens/s = forwards of all sequences / time."""
    import torch

    import llama_fp32_token_decode_b300 as l2

    torch.cuda.set_device(local)
    w = synth.workload("batched")
    cfg = synth.model_config(w)
    lens, prompts = synth.batch_inputs(w)
    B, steps, L = int(w["batch"]), int(w["steps"]), cfg["n_layers"]
    n_fwd = int(np.sum(lens + steps - 1))           # forwards of all sequences
    n_lock = int(lens.max()) + steps - 1            # lockstep steps
    blob = synth.make_blob(cfg, w["seed"])
    dec = l2.Decoder(cfg, blob)
    stream = torch.cuda.Stream()
    d_prompts = torch.tensor(prompts, dtype=torch.int32, device="cuda")
    d_out = torch.zeros((B, steps), dtype=torch.int32, device="cuda")

    def step():
        l2.l2_generate_batch_device(dec.h, d_prompts, lens, steps, d_out, stream)

    for _ in range(args.warmup):
        step()
    stream.synchronize()
    ref_tokens = d_out.cpu().numpy().copy()

    ms_max, clocks, _ = timed_steps(step, stream, args.steps, world, local)
    value = world * args.steps * n_fwd / (ms_max / 1e3)
    assert np.array_equal(d_out.cpu().numpy(), ref_tokens), "batched generation is not reproducible"

    # the same workload with every prompt taken by prefill passes (not the
    # headline: the measured step is the per-token decode)
    d_out_p = torch.zeros((B, steps), dtype=torch.int32, device="cuda")
    l2.l2_generate_batch_prefill_device(dec.h, d_prompts, lens, steps, d_out_p, stream)
    stream.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        l2.l2_generate_batch_prefill_device(dec.h, d_prompts, lens, steps, d_out_p, stream)
    e1.record(stream)
    e1.synchronize()
    ms_p = max_over_ranks(e0.elapsed_time(e1), world)
    agree = float(np.mean(d_out_p.cpu().numpy()[:, 0] == ref_tokens[:, 0]))
    with_prefill = {"value": world * args.steps * n_fwd / (ms_p / 1e3), "unit": "tok/s",
                    "ms_per_step": ms_p / args.steps,
                    "prompt_rows": int(np.sum(lens)), "lockstep_steps": steps - 1,
                    "first_token_agreement_with_lockstep": agree}

    # end to end: host prompts in, host tokens out
    h_prompts = torch.tensor(prompts, dtype=torch.int32).pin_memory().numpy()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        toks = dec.generate_batch(h_prompts, lens, steps)
    t_e2e = max_over_ranks(time.perf_counter() - t0, world)
    assert np.array_equal(toks, ref_tokens), "host and device batched entry points disagree"
    e2e = {"value": world * args.steps * n_fwd / t_e2e, "unit": "tok/s",
           "h2d_bytes_per_step": int(h_prompts.nbytes + lens.nbytes),
           "d2h_bytes_per_step": int(B * steps * 4)}

    # per-kernel times at the run's mean position, live, on the bench stream
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    p3, p3_source = tf32x3_peak(peaks)
    pos_mid = int(np.mean(lens)) - 1 + steps // 2
    per = {}
    for kind, name in BATCHED_KINDS.items():
        t = median_time(l2, dec.h, kind, pos_mid, 3 * L, stream)
        launches = {11: 1, 12: 1}.get(kind, L)
        shp = batched_gemm_shape(cfg, kind)
        flops = 2.0 * B * shp[0] * shp[1] if shp else 0.0
        per[kind] = {"name": name, "launch_ms": t, "launches_per_step": launches,
                     "ms_per_step": t * launches, "bytes": l2.l2_kernel_bytes(dec.h, kind, pos_mid),
                     "flops": flops}
    total_ms = sum(v["ms_per_step"] for v in per.values())
    dom = max(per, key=lambda k: per[k]["ms_per_step"])
    dk = per[dom]
    if dk["flops"] > 0:
        ach = dk["flops"] / (dk["launch_ms"] / 1e3) / 1e12
        roofline = {"bound": "tensor", "achieved": ach, "peak": p3, "unit": "TFLOP/s",
                    "frac": ach / p3, "traffic": None}
    else:
        ach = dk["bytes"] / (dk["launch_ms"] / 1e3) / 1e9
        roofline = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                    "frac": ach / hbm,
                    "traffic": profiled_battn_traffic(dk["bytes"]) if dom == 7 else None}
    roofline.update({"kernel": dk["name"], "launch_ms": dk["launch_ms"],
                     "share_of_kernel_time": dk["ms_per_step"] / total_ms,
                     "peak_source": (p3_source if dk["flops"] > 0
                                     else f"{peak_kind} hbm_gbs (copy)")})
    g_flops = sum(v["flops"] * v["launches_per_step"] for v in per.values())
    g_ms = sum(v["ms_per_step"] for v in per.values() if v["flops"] > 0)
    gemm_phase = {"achieved": g_flops / (g_ms / 1e3) / 1e12, "peak": p3, "unit": "TFLOP/s",
                  "frac": g_flops / (g_ms / 1e3) / 1e12 / p3, "flops_per_step": g_flops,
                  "ms_per_step": g_ms, "peak_source": p3_source,
                  "measured_fp32_gemm_peaks": measured_fp32_peaks()}
    attn = per[7]
    attn_roof = {"achieved": attn["bytes"] / (attn["launch_ms"] / 1e3) / 1e9, "peak": hbm,
                 "unit": "GB/s", "frac": attn["bytes"] / (attn["launch_ms"] / 1e3) / 1e9 / hbm,
                 "pos": pos_mid}
    kernels = {v["name"]: round(v["ms_per_step"] / total_ms, 4) for v in per.values()}
    bound_s, gemm_bound_s = batched_run_bound(cfg, lens, steps, B, hbm, p3)
    run_s = ms_max / args.steps / 1e3
    step_roof = {"bound_ms": bound_s * 1e3, "gemm_phases_bound_ms": gemm_bound_s * 1e3,
                 "measured_ms": run_s * 1e3, "frac": bound_s / run_s,
                 "roofline_tok_s": n_fwd / bound_s,
                 "note": "sum over lockstep steps of max(fp32 weights / HBM, GEMM FLOPs / "
                         "3xTF32 peak) + active rows' KV bytes / HBM"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nf = args.cpu_forwards or 60
        import oracle
        m = oracle.Model(cfg, blob)
        tok = int(prompts[0])
        t0 = time.perf_counter()
        for p in range(nf):
            lg = m.forward(tok, p)
            tok = int(prompts[p + 1]) if p + 1 < lens[0] else int(np.argmax(lg))
        dt = time.perf_counter() - t0
        m.close()
        cpu = {"value": nf / dt, "unit": "tok/s", "cores": 1, "kind": "oracle",
               "sample": f"sequence 0 of the batched workload, first {nf} forwards, "
                         f"single-threaded C oracle (-O2, no fast-math); the oracle decodes "
                         f"sequences one after another"}
    dec.close()
    line = {"metric": METRIC_BATCHED, "value": value, "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (random-init N(0,0.02) weights, seeded prompts and lengths)",
            "config": {"workload": "batched", "global_batch": world * B, "dim": cfg["dim"],
                       "n_layers": L, "n_heads": cfg["n_heads"],
                       "hidden_dim": cfg["hidden_dim"], "vocab_size": cfg["vocab_size"],
                       "seq_len": cfg["seq_len"], "prompt_lens": "U[1,128] seed 4",
                       "generated_per_sequence": steps, "forwards_per_step": n_fwd,
                       "lockstep_steps": n_lock, "parallelism": f"replicas{world}",
                       "l2": "inputs larger than L2 (KV caches %.1f GB)" % (
                           B * 2 * L * cfg["seq_len"] * cfg["dim"] * 4 / 1e9)},
            "roofline": roofline, "gemm_phase_roofline": gemm_phase,
            "attention_roofline": attn_roof, "kernel_time_shares": kernels,
            "step_roofline": step_roof, "with_prefill": with_prefill,
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": args.steps * (1 + n_lock * (2 + 5 * L + 1))}
    if compact:
        for k in ("steps", "warmup", "higher_is_better", "scaling", "vs_baseline", "data",
                  "n_gpus"):
            line.pop(k, None)
    return line


def run_kernel_only(args):
    """Small case of one kernel for profilers: the workload's shapes with fewer
    layers and a 512-position cache (a few GB on the device), one warm-up launch
    and two timed launches of the chosen kind."""
    import torch

    import llama_fp32_token_decode_b300 as l2
    torch.cuda.set_device(0)
    w = synth.workload(args.workload)
    cfg = synth.model_config(w)
    if args.layers:
        cfg["n_layers"] = args.layers
    if args.workload == "7b" and args.kernel_only in (8, 9, 10):
        # the GEMMs of the 7B prefill pass: its prompt's rows, one KV cache
        cfg["max_prefill"] = w["n_prompt"]
    # a short cache keeps the case to a few GB (batched: 256 caches)
    cfg["seq_len"] = min(cfg["seq_len"], 384 if cfg.get("max_batch", 1) > 1 else 512)
    blob = synth.make_blob(cfg, w["seed"])
    with l2.Decoder(cfg, blob) as dec:
        pos = min(300, cfg["seq_len"] - 1)
        ms = l2.l2_time_kernel(dec.h, args.kernel_only, pos, 2)
        b = l2.l2_kernel_bytes(dec.h, args.kernel_only, pos)
    print(json.dumps({"kernel": l2.KERNEL_KINDS[args.kernel_only], "workload": args.workload,
                      "layers": cfg["n_layers"], "pos": pos, "launch_ms": ms,
                      "algorithmic_bytes": b, "GB/s": b / ms / 1e6}), flush=True)
    return 0


def main():
    args = parse_args()
    if args.kernel_only is not None:
        return run_kernel_only(args)
    world, rank, local = dist_setup(args)
    if args.gpus != world and world > 1:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE {world}")
    if args.impl == "reference":
        rc = run_reference(args, world, rank)
    elif args.workload == "batched":
        line = run_ours_batched(args, world, rank, local)
        if rank == 0:
            print(json.dumps(line), flush=True)
        rc = 0
    else:
        rc = run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
