#!/usr/bin/env python
"""Throughput benchmark of the B300 GPT-2 training step.

One step = forward (with the mean cross-entropy loss) + zero_grad + backward +
AdamW over the whole model, through the library's C ABI.  The default
workload is GPT-2 124M at B=16, T=1024 in bf16 with fp32 master weights: the
throughput configuration (5 warm-up + 50 timed steps, AdamW lr 6e-4,
wd 0.1, Zipf(1.1) token stream, a fresh batch per step).  Weights are the
library's own random GPT-2 init; data are synthetic (no dataset is used).

Prints ONE JSON line (rank 0).  Keys:
  value / ms_per_step   tokens/s over all ranks, inputs resident in HBM,
                        timed with CUDA events on the model's stream
  e2e                   the same metric through gpt2_forward_host (pinned
                        host token buffers copied in every step, the loss
                        read back every step)
  roofline              the kernel class with the largest share of the step,
                        timed live with CUDA events inside the timed region:
                        algorithmic work per launch / average launch duration
                        against the measured peak
  mfu                   one GPU's tokens/s x algorithmic FLOPs per token over the
                        measured bf16 burst and sustained peaks; six_n: the same with
                        the 6 x parameters convention, for comparison only
  cpu_baseline          the CPU oracle timed on this host on a bounded sample
  clocks                nvidia-smi samples taken during the timed region
  gpu_launches          kernel launches of the library inside the timed region

--impl reference times the CPU oracle itself (the only other implementation
of this step) on bounded samples of the same workload.

--mode fp8 measures the E4M3 matmuls (gpt2_fp8_matmul) on the five forward
products of GPT-2 124M at M = B*T = 16384 rows (qkv, attproj, fc, fcproj,
tied head) with bf16 outputs: value = their total FLOPs / total time
(each product timed alone with CUDA events, L2 flushed before each), the
roofline against twice the measured bf16 peak (the nominal fp8 : bf16
tensor ratio).

--mode oracle times one full step of the CPU oracle on the tiny and
char-level configurations and on GPT-2 124M at B=4, T=1024 (tokens/s per
configuration, the host's CPU model and thread count); it uses no GPU.

--mode decode measures generation with the key/value cache instead: GPT-2
124M, B=16 sequences, a 512-token prompt per sequence run through one
forward (the prefill), then one gpt2_decode_step per new token (temperature
1.0, uniforms from a fixed seed).  value = generated tokens/s over the timed
decode steps; the roofline is the whole decode step against the HBM copy
peak (its algorithmic bytes: the bf16 weights read once, the cached keys and
values of rows 0..pos read once, the new cache row and the scores written).
"""
import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GPT-2 124M train tokens/sec (fwd+bwd+AdamW) on 1 B300; MFU vs bf16 peak"

WORKLOADS = {
    # the throughput configuration: B=16, T=1024, Zipf(1.1) tokens, 50 timed steps
    "gpt2-124M-B16-T1024": dict(L=12, C=768, NH=12, V=50257, Vp=50304, maxT=1024, B=16, T=1024,
                                dist="zipf", lr=6e-4, wd=0.1),
    "gpt2-124M-B4-T1024": dict(L=12, C=768, NH=12, V=50257, Vp=50304, maxT=1024, B=4, T=1024,
                               dist="uniform", lr=6e-4, wd=0.1),
    "gpt2-350M-B8-T1024": dict(L=24, C=1024, NH=16, V=50257, Vp=50304, maxT=1024, B=8, T=1024,
                               dist="uniform", lr=6e-4, wd=0.1),
    # the 124M model on a small batch: the size used for ncu captures
    "gpt2-124M-B2-T1024": dict(L=12, C=768, NH=12, V=50257, Vp=50304, maxT=1024, B=2, T=1024,
                               dist="zipf", lr=6e-4, wd=0.1),
    # two 124M layers at the throughput batch: the attention and layer kernels
    # see the throughput shapes, the device holds ~4 GB (ncu captures)
    "gpt2-124M-L2-B16-T1024": dict(L=2, C=768, NH=12, V=50257, Vp=50304, maxT=1024, B=16, T=1024,
                                   dist="zipf", lr=6e-4, wd=0.1),
}
DEFAULT_WORKLOAD = "gpt2-124M-B16-T1024"
DECODE_METRIC = "GPT-2 124M generated tokens/sec with a key/value cache (B=16 sequences) on 1 B300"
DECODE = dict(L=12, C=768, NH=12, V=50257, Vp=50304, maxT=1024, B=16, T=1024, prompt=512, temperature=1.0)
BETAS, EPS = (0.9, 0.999), 1e-8
L2_BYTES = 126 * 2 ** 20


def flops_per_token(w):
    """Algorithmic FLOPs per token: 3 x (matmuls + causal attention), forward
    = 2 L (3C^2 + C^2 + 4C^2 + 4C^2) + 2 C Vp + 2*2 L C (T/2)."""
    L, C, Vp, T = w["L"], w["C"], w["Vp"], w["T"]
    return 3.0 * (2 * L * 12 * C * C + 2 * C * Vp + 4 * L * C * (T / 2))


def num_params(w):
    """Parameters without the vocabulary padding: wte, wpe, L blocks of
    12 C^2 + 13 C (four Linears with biases, two LayerNorms) and the final
    LayerNorm."""
    L, C = w["L"], w["C"]
    return w["V"] * C + w["maxT"] * C + L * (12 * C * C + 13 * C) + 2 * C


def mfu_report(tokens_per_s_per_gpu, w, peaks):
    """MFU of one GPU's throughput against the bf16 burst and sustained
    peaks with the algorithmic FLOPs per token; the common 6N convention
    (6 x parameters per token, no attention scores) beside it, for
    comparison only."""
    ftok = flops_per_token(w)
    f6n = 6.0 * num_params(w)
    r = lambda f, peak: round(tokens_per_s_per_gpu * f / (peak * 1e12), 4)  # noqa: E731
    return dict(vs_bf16_burst=r(ftok, peaks["bf16"]), vs_bf16_sustained=r(ftok, peaks["bf16_sustained"]),
                flops_per_token=ftok, peak_source=peaks["source"],
                six_n=dict(flops_per_token=f6n, vs_bf16_burst=r(f6n, peaks["bf16"]),
                           vs_bf16_sustained=r(f6n, peaks["bf16_sustained"])))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm_gbs=6400.0, bf16=1800.0, bf16_sustained=1400.0, source="fallback")


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while running (reading only)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_id)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        sm.sort()
        return dict(sm_mhz=sm[len(sm) // 2], sm_max_mhz=max(mx), reasons=sorted(reasons),
                    samples=len(sm))


# ---------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_ms, local_tokens, world, backend_device=None):
    """Max of the per-rank elapsed times and sum of tokens over ranks:
    value = all tokens / slowest rank's time."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([local_ms], dtype=torch.float64, device=backend_device)
        n = torch.tensor([float(local_tokens)], dtype=torch.float64, device=backend_device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(n, op=dist.ReduceOp.SUM)
        local_ms, local_tokens = float(t.item()), float(n.item())
    return local_ms, local_tokens, local_tokens / (local_ms / 1000.0)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- CPU oracle
def oracle_sample_rate(w, B, T, steps, seed=7, warmup=0):
    """Tokens/s of the CPU oracle on `steps` full steps (fwd + bwd + AdamW)
    of the workload's model on a B x T sample."""
    import numpy as np

    import oracle
    from transformer_lm_step_gpt_b300 import synthetic
    cores = oracle.set_threads(len(os.sched_getaffinity(0)))
    cfg = oracle.cfg8(w["L"], w["C"], w["NH"], w["V"], w["Vp"], w["maxT"], B, T)
    tab = oracle.param_table(cfg)
    p = synthetic.params(tab, w["L"], w["C"], w["V"], seed, kind="gpt2_init")
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    for i in range(warmup):
        tok, tgt = synthetic.batch(seed + 100 + i, B, T, w["V"], w["dist"])
        oracle.step(cfg, p, m, v, tok, tgt, w["lr"], BETAS[0], BETAS[1], EPS, w["wd"], i + 1)
    t0 = time.perf_counter()
    for i in range(steps):
        tok, tgt = synthetic.batch(seed + i, B, T, w["V"], w["dist"])
        oracle.step(cfg, p, m, v, tok, tgt, w["lr"], BETAS[0], BETAS[1], EPS, w["wd"], warmup + i + 1)
    dt = time.perf_counter() - t0
    return steps * B * T / dt, cores, dt


def cpu_baseline(w):
    # bounded sample: one sequence of 128 tokens per step, up to ~20 s of CPU work
    B, T = 1, 128
    rate, cores, dt = oracle_sample_rate(w, B, T, 1)
    steps = max(1, min(8, int(20.0 / max(dt, 1e-3))))
    if steps > 1:
        rate, cores, dt = oracle_sample_rate(w, B, T, steps)
    return dict(value=rate, unit="tokens/s", cores=cores, kind="oracle",
                sample="%d full training step(s) (fwd+bwd+AdamW over all %s parameters) on B=%d, T=%d "
                       "of the %s model, %.1f s" % (steps, "124M" if w["L"] == 12 else "350M", B, T,
                                                    "GPT-2", dt))


# ---------------------------------------------------------------- helpers
def source_digest(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(kernel_class):
    """DRAM traffic per launch from a committed ncu summary, if the kernel's
    sources are unchanged since it was captured."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(kernel_class)
        if e and source_digest(e["sources"]) == e["digest"]:
            return float(e["bytes_per_launch"])
    except Exception:
        pass
    return None


def gpu_uuid(dev):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev)


# ---------------------------------------------------------------- our arm
def run_ours(args, w, world, rank, local):
    import numpy as np
    import torch

    import transformer_lm_step_gpt_b300 as tl
    from transformer_lm_step_gpt_b300 import synthetic

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    B, T = w["B"], w["T"]
    stream = torch.cuda.Stream(device=dev)
    m = tl.Model(w["L"], w["C"], w["NH"], w["V"], w["Vp"], w["maxT"], B, T, precision="bf16",
                 seed=1337 + rank, stream=stream)
    W, K = args.warmup, args.steps
    # every step gets a fresh batch of the token stream; all batches are made
    # and copied to the device before the timed region
    batches_h = [synthetic.batch(1338 + rank * 100003 + i, B, T, w["V"], w["dist"]) for i in range(W + K)]
    with torch.cuda.stream(stream):
        batches_d = [(torch.from_numpy(t).to(dev), torch.from_numpy(g).to(dev)) for t, g in batches_h]
    stream.synchronize()
    lr, wd = w["lr"], w["wd"]
    t_step = [0]

    def step(tok, tgt, host=False):
        t_step[0] += 1
        if host:
            m.forward_host(tok, tgt, sync=False)
        else:
            m.forward(tok, tgt, sync=False)
        m.zero_grad()
        m.backward()
        m.adamw_step(lr, BETAS[0], BETAS[1], EPS, wd, t_step[0])

    # warm-up; the last warm-up step is timed per kernel class to find the
    # class with the largest share of the step
    for i in range(W):
        if i == W - 1:
            m.profile_enable("all")
            m.profile_reset()
        step(*batches_d[i])
    prof = m.profile_read()
    m.profile_enable(None)
    step_ms_prof = sum(r["ms"] for r in prof)
    top = max(prof, key=lambda r: r["ms"])
    breakdown = {r["name"]: round(r["ms"], 4) for r in prof if r["launches"]}

    # timed region: exactly K steps, barrier + synchronize on both sides
    m.profile_enable([top["name"]])
    m.profile_reset()
    clocks = ClockSampler(gpu_uuid(local))
    clocks.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    n0 = m.launch_count
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K):
        step(*batches_d[W + i])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    local_ms = e0.elapsed_time(e1)
    launches = m.launch_count - n0
    kprof = [r for r in m.profile_read() if r["name"] == top["name"]][0]
    m.profile_enable(None)
    loss_last = m.read_loss()
    total_ms, total_tokens, value = aggregate(local_ms, K * B * T, world, dev)
    ms_per_step = total_ms / K

    # end to end through the host entry point: pinned host ids copied in and
    # the loss read back every step
    pinned = [(torch.from_numpy(t).pin_memory(), torch.from_numpy(g).pin_memory()) for t, g in batches_h]
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(K):
        tok, tgt = pinned[W + i]
        step(tok, tgt, host=True)
        m.read_loss()
    t1 = time.perf_counter()
    barrier(world)
    _, _, e2e_value = aggregate((t1 - t0) * 1000.0, K * B * T, world, dev)

    peaks = load_peaks()
    tensor = top["unit"] == "flop"
    avg_ms = kprof["ms"] / max(kprof["launches"], 1)
    work_per_launch = kprof["work"] / max(kprof["launches"], 1)
    if tensor:
        achieved = work_per_launch / (avg_ms / 1e3) / 1e12
        peak = peaks["bf16_sustained"]
    else:
        achieved = work_per_launch / (avg_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
    roofline = dict(bound="tensor" if tensor else "hbm", achieved=round(achieved, 2), peak=peak,
                    unit="TFLOP/s" if tensor else "GB/s", frac=round(achieved / peak, 4),
                    traffic=load_traffic(top["name"]), kernel=top["name"],
                    launches_per_step=kprof["launches"] / K, avg_launch_ms=round(avg_ms, 4),
                    work_per_launch=work_per_launch, work_unit=top["unit"],
                    peak_source="%s %s" % (peaks["source"], "bf16_tflops_sustained" if tensor else "hbm_gbs"),
                    share_of_step=round(kprof["ms"] / K / ms_per_step, 4))
    out = dict(metric=METRIC, value=round(value, 1), unit="tokens/s", n_gpus=world, steps=K, warmup=W,
               ms_per_step=round(ms_per_step, 4), higher_is_better=True, scaling="weak",
               vs_baseline=None, dtype="bf16",
               data="synthetic: Zipf(1.1)/uniform int32 token stream from a fixed seed, a fresh "
                    "batch per step; random GPT-2 init weights (no dataset, no checkpoint)",
               config=dict(workload=args.workload, global_batch=B * world, seq_len=T,
                           parallelism="replicas only" if world > 1 else "single GPU",
                           layers=w["L"], channels=w["C"], heads=w["NH"], vocab=w["V"], padded_vocab=w["Vp"],
                           token_dist=w["dist"], lr=lr, weight_decay=wd, betas=list(BETAS), eps=EPS,
                           seeds=dict(build=1337 + rank, token_batches="1338 + 100003 * rank + step index"),
                           l2="no flush: each step streams ~%.1f GB of weights, activations and optimizer "
                              "state (> 126 MB L2)" % (step_bytes(w) / 1e9)),
               mfu=mfu_report(value / world, w, peaks),
               roofline=roofline,
               e2e=dict(value=round(e2e_value, 1), unit="tokens/s", h2d_bytes_per_step=2 * B * T * 4,
                        d2h_bytes_per_step=4),
               gpu_launches=launches,
               clocks=clk,
               kernels_ms_per_step=breakdown,
               loss_last_step=loss_last)
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w)
    elif world > 1:
        out["cpu_baseline"] = None
    m.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return out if rank == 0 else None


def step_bytes(w):
    """Rough bytes one step moves (weights, optimizer state, activations)."""
    L, C, B, T, Vp = w["L"], w["C"], w["B"], w["T"], w["Vp"]
    n = Vp * C + w["maxT"] * C + L * 12 * C * C
    acts = B * T * (L * (4 * 2 * C + 2 * 16 * C) + 2 * Vp)
    return 30 * n + 3 * acts


# ---------------------------------------------------------------- decode mode
def decode_step_bytes(d, pos):
    """Algorithmic bytes of one decode step at position pos: every input read
    once (bf16 weight matrices, fp32 biases and LayerNorm parameters, the
    token and position embedding rows, the cached keys and values of rows
    0..pos-1), every output written once (the new cache row of q, k, v); the
    scores and the per-row activations are intermediates."""
    L, C, Vp, B = d["L"], d["C"], d["Vp"], d["B"]
    matrices = 2 * (Vp * C + L * 12 * C * C)
    small = 4 * (L * 13 * C + 2 * C) + 4 * (B + 1) * C
    kv_read = 2 * L * B * pos * 2 * C
    new_row = 2 * L * B * 3 * C
    return matrices + small + kv_read + new_row


def run_decode(args, world, rank, local):
    import numpy as np
    import torch

    import transformer_lm_step_gpt_b300 as tl

    d = DECODE
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B, T, P = d["B"], d["T"], d["prompt"]
    stream = torch.cuda.Stream(device=dev)
    m = tl.Model(d["L"], d["C"], d["NH"], d["V"], d["Vp"], d["maxT"], B, T, precision="bf16",
                 seed=1337 + rank, stream=stream)
    W, K = args.warmup, args.steps
    if P - 1 + W + K > T:
        raise SystemExit("decode mode: prompt + warm-up + steps must fit in %d positions" % T)
    rng = np.random.default_rng(77 + rank)
    prompt = np.zeros((B, T), np.int32)
    prompt[:, :P] = rng.integers(0, d["V"], (B, P))
    u = rng.random((W + K, B)).astype(np.float32)
    with torch.cuda.stream(stream):
        tok_d = torch.from_numpy(prompt).to(dev)
        seq = torch.empty((W + K + 1, B), dtype=torch.int32, device=dev)
        seq[0] = tok_d[:, P - 1]
        u_d = torch.from_numpy(u).to(dev)
    stream.synchronize()
    m.forward(tok_d, None, sync=False)
    for i in range(W):
        m.decode_step(seq[i], P - 1 + i, d["temperature"], u_d[i], out=seq[i + 1])
    m.profile_enable("all")
    m.profile_reset()
    clocks = ClockSampler(gpu_uuid(local))
    clocks.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    n0 = m.launch_count
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(W, W + K):
        m.decode_step(seq[i], P - 1 + i, d["temperature"], u_d[i], out=seq[i + 1])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    local_ms = e0.elapsed_time(e1)
    launches = m.launch_count - n0
    prof = m.profile_read()
    m.profile_enable(None)
    total_ms, _, value = aggregate(local_ms, K * B, world, dev)
    ms_per_step = total_ms / K
    # profiling events around every launch stretch the step a little: time
    # the same steps again without them for the reported value
    m.forward(tok_d, None, sync=False)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0.record(stream)
    h0 = time.perf_counter()
    for i in range(W, W + K):
        m.decode_step(seq[i], P - 1 + i, d["temperature"], u_d[i], out=seq[i + 1])
    host_ms = (time.perf_counter() - h0) * 1e3 / K  # time to enqueue one step
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    total_ms, _, value = aggregate(e0.elapsed_time(e1), K * B, world, dev)
    ms_per_step = total_ms / K
    by = sum(decode_step_bytes(d, P - 1 + i) for i in range(W, W + K)) / K
    peaks = load_peaks()
    achieved = by / (ms_per_step / 1e3) / 1e9
    breakdown = {r["name"]: round(r["ms"] / K, 4) for r in prof if r["launches"]}
    # end to end through Model.generate: prompt copied in, prefill forward,
    # K new tokens, all tokens read back
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    m.generate(prompt[:, :P], K, temperature=d["temperature"], uniforms=u[:K])
    e2e = K * B / (time.perf_counter() - t0) * world
    out = dict(metric=DECODE_METRIC, value=round(value, 1), unit="tokens/s", n_gpus=world, steps=K, warmup=W,
               ms_per_step=round(ms_per_step, 4), higher_is_better=True, scaling="weak", vs_baseline=None,
               dtype="bf16", data="synthetic: uniform prompt ids, random GPT-2 init weights, uniforms from a fixed seed",
               config=dict(workload="gpt2-124M-decode-B16-P512", batch=B, prompt=P, cache_rows=T,
                           temperature=d["temperature"], mode="decode",
                           l2="no flush: each step reads the 0.25 GB of bf16 weights and the cache (> 126 MB L2)"),
               roofline=dict(bound="hbm", achieved=round(achieved, 1), peak=peaks["hbm_gbs"], unit="GB/s",
                             frac=round(achieved / peaks["hbm_gbs"], 4), traffic=None, kernel="decode step (all kernels)",
                             bytes_per_step=by, peak_source="%s hbm_gbs" % peaks["source"]),
               e2e=dict(value=round(e2e, 1), unit="tokens/s", h2d_bytes_per_step=round(B * P * 4 / K + B * 4, 1),
                        d2h_bytes_per_step=B * 4,
                        note="Model.generate: prefill forward + %d decode steps, prompt in and tokens out" % K),
               gpu_launches=launches, clocks=clk, kernels_ms_per_step=breakdown,
               host_enqueue_ms_per_step=round(host_ms, 4))
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = decode_cpu_baseline(d)
    m.close()
    return out if rank == 0 else None


def decode_cpu_baseline(d):
    import numpy as np

    import oracle
    cfg = oracle.cfg8(d["L"], d["C"], d["NH"], d["V"], d["Vp"], d["maxT"], 1, 8)
    p = oracle.init_params(cfg, 1337)
    prompt = np.arange(1, 9, dtype=np.int32).reshape(1, 8)
    n_new = 4
    t0 = time.perf_counter()
    oracle.generate(cfg, p, prompt, n_new, 1.0, np.full((n_new, 1), 0.5))
    dt = time.perf_counter() - t0
    return dict(value=n_new / dt, unit="tokens/s", cores=1, kind="oracle",
                sample="one sequence: an 8-token prompt and %d new tokens through the oracle's incremental "
                       "forward (fp64, one thread per sequence), %.1f s" % (n_new, dt))


# ---------------------------------------------------------------- fp8 mode
FP8_METRIC = "GPT-2 124M forward matmuls in FP8 (E4M3, per-tensor scales) TFLOP/s on 1 B300"
FP8_SHAPES = [("qkv", 2304, 768), ("attproj", 768, 768), ("fc", 3072, 768), ("fcproj", 768, 3072),
              ("head", 50304, 768)]


def run_fp8(args):
    import numpy as np
    import torch

    import transformer_lm_step_gpt_b300 as tl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    M = 16384
    g = torch.Generator(device=dev).manual_seed(5)
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
    ops = []
    for name, N, K in FP8_SHAPES:
        a = torch.randn((M, K), generator=g, device=dev)
        w = torch.randn((N, K), generator=g, device=dev) * 0.02
        qa, sa = tl.fp8_quantize(a)
        qw, sw = tl.fp8_quantize(w)
        ops.append((name, N, K, qa, sa, qw, sw))
    torch.cuda.synchronize()
    W, Kst = args.warmup, args.steps
    per = {}
    clocks = ClockSampler(gpu_uuid(0))
    clocks.start()
    for name, N, K, qa, sa, qw, sw in ops:
        for _ in range(W):
            tl.fp8_matmul(qa, sa, qw, sw, out_dtype=torch.bfloat16)
        ms = 0.0
        for _ in range(Kst):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            tl.fp8_matmul(qa, sa, qw, sw, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize()
            ms += e0.elapsed_time(e1)
        per[name] = dict(N=N, K=K, ms=ms / Kst, tflops=2.0 * M * N * K / (ms / Kst / 1e3) / 1e12)
    clk = clocks.stop()
    tl.fp8_check()
    flops = sum(2.0 * M * v["N"] * v["K"] for v in per.values())
    tot_ms = sum(v["ms"] for v in per.values())
    value = flops / (tot_ms / 1e3) / 1e12
    peaks = load_peaks()
    peak = 2.0 * peaks["bf16"]
    top = max(per, key=lambda k: per[k]["ms"])
    # end to end: fp32 activations from pinned host memory, quantised and
    # multiplied on the device, the bf16 result read back (weights resident)
    name, N, K, _, _, qw, sw = [o for o in ops if o[0] == "fc"][0]
    a_h = torch.randn((M, K)).pin_memory()
    o_h = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(Kst):
        a_d = a_h.to(dev, non_blocking=True)
        qa, sa = tl.fp8_quantize(a_d)
        o_h.copy_(tl.fp8_matmul(qa, sa, qw, sw, out_dtype=torch.bfloat16), non_blocking=True)
    torch.cuda.synchronize()
    e2e = 2.0 * M * N * K * Kst / (time.perf_counter() - t0) / 1e12
    out = dict(metric=FP8_METRIC, value=round(value, 1), unit="TFLOP/s", n_gpus=1, steps=Kst, warmup=W,
               ms_per_step=round(tot_ms, 4), higher_is_better=True, scaling="weak", vs_baseline=None,
               dtype="e4m3", data="synthetic: normal activations, N(0, 0.02) weights, quantised with per-tensor scales",
               config=dict(workload="gpt2-124M-forward-matmuls-M16384-fp8", rows=M, mode="fp8",
                           products={k: [v["N"], v["K"]] for k, v in per.items()},
                           l2="flushed (256 MB write) before every timed product"),
               roofline=dict(bound="tensor", achieved=round(per[top]["tflops"], 1), peak=peak, unit="TFLOP/s",
                             frac=round(per[top]["tflops"] / peak, 4), traffic=None, kernel="gemm_tc_pair_kernel<F8> (%s)" % top,
                             peak_source="%s bf16_tflops x 2 (nominal fp8 : bf16 ratio)" % peaks["source"]),
               e2e=dict(value=round(e2e, 1), unit="TFLOP/s", h2d_bytes_per_step=M * K * 4, d2h_bytes_per_step=M * N * 2,
                        note="fc shape: fp32 activations in from pinned memory, quantise, matmul, bf16 out"),
               gpu_launches=len(per) * Kst, clocks=clk,
               products={k: dict(ms=round(v["ms"], 4), tflops=round(v["tflops"], 1)) for k, v in per.items()})
    if not args.no_cpu_baseline:
        import oracle
        rng = np.random.default_rng(0)
        qa = rng.integers(0, 0x7E, (8, 768)).astype(np.uint8)
        qb = rng.integers(0, 0x7E, (768, 768)).astype(np.uint8)
        t0 = time.perf_counter()
        oracle.fp8_matmul(qa, 1.0, qb, 1.0)
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = dict(value=2.0 * 8 * 768 * 768 / dt / 1e12, unit="TFLOP/s", cores=oracle.set_threads(0),
                                   kind="oracle", sample="8 x 768 x 768 product of the oracle's fp8_matmul, %.2f s" % dt)
    return out


# ---------------------------------------------------------------- reference arm
def run_reference(args, w, world, rank):
    if rank != 0:
        return None
    # each step: one full training step of the oracle on a bounded sample
    # (one sequence of 32 tokens of the same model), so that W + K steps end
    # within a few minutes
    B, T = 1, 32
    rate, cores, dt = oracle_sample_rate(w, B, T, args.steps, warmup=args.warmup)
    sample = ("per step: one full oracle training step (fwd+bwd+AdamW over all parameters) on B=%d, "
              "T=%d of the %s workload" % (B, T, args.workload))
    model = "gpt2-124M" if w["L"] == 12 else ("gpt2-350M" if w["L"] == 24 else "gpt2-L%d" % w["L"])
    return dict(impl="reference", metric=METRIC, value=round(rate, 3), unit="tokens/s", n_gpus=world,
                steps=args.steps, warmup=args.warmup, ms_per_step=round(dt / args.steps * 1000, 2),
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f32",
                data="synthetic: same token stream recipe and GPT-2 init as our arm",
                config=dict(workload="%s-B%d-T%d" % (model, B, T), sample_of=args.workload, global_batch=B,
                            seq_len=T, parallelism="CPU oracle, rank 0 only", cpu_model=cpu_model()),
                cpu_baseline=dict(value=round(rate, 3), unit="tokens/s", kind="oracle", cores=cores,
                                  sample=sample),
                e2e=dict(value=round(rate, 3), unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


# the method's configurations whose full steps the oracle runs (one step each)
ORACLE_CONFIGS = {
    "tiny-fp32 (L2 C64 NH4 T32 B4 V256)": dict(L=2, C=64, NH=4, V=256, Vp=256, maxT=32, B=4, T=32,
                                              dist="uniform", lr=1e-4, wd=0.0),
    "char (L8 C128 NH8 T64 B32 V1000)": dict(L=8, C=128, NH=8, V=1000, Vp=1000, maxT=64, B=32, T=64,
                                            dist="zipf", lr=3e-4, wd=0.1),
    "gpt2-124M-B4-T1024": WORKLOADS["gpt2-124M-B4-T1024"],
}


def run_oracle_timing(args):
    """One full training step (fwd + bwd + AdamW) of the CPU oracle on each
    configuration the oracle can finish: the tiny and char-level models and
    GPT-2 124M at B=4, T=1024, with the host's CPU model and thread count."""
    out = dict(mode="oracle", metric="CPU oracle training tokens/sec, one full step per configuration",
               unit="tokens/s", cpu_model=cpu_model(), configs={})
    for name, w in ORACLE_CONFIGS.items():
        rate, cores, dt = oracle_sample_rate(w, w["B"], w["T"], 1)
        out["configs"][name] = dict(tokens=w["B"] * w["T"], seconds=round(dt, 3), tokens_per_s=round(rate, 2),
                                    flops_per_token=flops_per_token(w),
                                    gflops_per_s=round(rate * flops_per_token(w) / 1e9, 2))
        out["cores"] = cores
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mode", choices=["train", "decode", "fp8", "oracle"], default="train")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if world != args.gpus and world > 1:
        print("warning: WORLD_SIZE=%d but --gpus %d" % (world, args.gpus), file=sys.stderr)
    w = WORKLOADS[args.workload]
    if args.mode == "oracle":
        out = run_oracle_timing(args) if rank == 0 else None
    elif args.mode == "decode" and args.impl == "ours":
        out = run_decode(args, world, rank, local)
    elif args.mode == "fp8" and args.impl == "ours":
        out = run_fp8(args) if rank == 0 else None
    else:
        out = run_reference(args, w, world, rank) if args.impl == "reference" else run_ours(args, w, world, rank, local)
    if out is not None and rank == 0:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
