"""Benchmark of one layer-streamed NF4 LoRA training step on one B300.

Workload (default): the Llama-3.1-8B-shaped stack (32 layers, hidden 4096, 32/8
heads, head_dim 128, SwiGLU 14336, vocabulary 128256 untied, RoPE theta 5e5) with an
NF4 base held in pinned host RAM and LoRA r=16 on q_proj/v_proj, trained with DPO
(beta 0.1) on one (chosen, rejected) pair: a shared 256-token prompt and 256-token
responses, so each pass carries 2 x 512 tokens.  One step = policy forward (adapter
on, activation store kept) and reference forward (same streamed base, adapter off)
in one shared sweep of the layers, DPO loss, streamed backward, LoRA gradient
gather, AdamW step on the adapters (fp32 master weights).  Weights and tokens are seeded
synthetic draws (N(0, 0.02) base, N(0, 0.01) adapters, uniform tokens).

Prints ONE JSON line (rank 0).  value = policy tokens per second with the batch
already on the device; e2e = the same through Stack.train_step from pinned host
buffers (batch upload and loss read-back inside the timed region).  Each step
streams about 8 GB of NF4 weights, far more than the 126 MB L2, so no flush is
needed between steps.  Per-kernel times (the roofline object) come from a second
run of the same steps with every kernel bracketed by CUDA events.  The `sft` object
is the SFT step at the same shape and batch (both sequences, every position a
target) on the same pinned base, with the DPO/SFT ratios of layer reads and peak
device bytes beside the ones the pages quote (1.52x and 0.914x).

--impl reference times the CPU oracle (fp64) on a bounded sample of the same
workload: each timed step is one decoder layer (policy forward + backward,
reference forward) plus 1/L of the vocabulary head, i.e. 1/L of a training step.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "train tokens/s streamed NF4 LoRA (8B shape, SFT+DPO); H2D GB/s; % roofline"
# DRAM bytes (read + write) per algorithmic byte of each NF4 GEMM class, from one ncu
# capture of the class's largest launch in the step (8B gate|up products: forward 2048 rows
# on paired split tiles, input gradient 1024 rows on the split schedule), in the build the
# step runs.  It scales the class's algorithmic bytes per launch to the reported traffic;
# None whenever that kernel has changed since the capture (the traffic is then null).
GEMM_TRAFFIC_PER_ALG_BYTE = {"gemm_fwd": (85.9 + 105.9) / 200.3,    # gate|up forward, 2048 rows, paired split
                             "gemm_dx": (449.1 + 17.8) / 141.6}     # gate|up input gradient, 1024 rows, split
UNIT = "tokens/s"
NF4_BYTES_PER_PARAM = 0.5625


# ----------------------------------------------------------------------------- helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend)


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """Largest value of x over all ranks (the job ends when the slowest rank ends)."""
    if ws <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", j["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples (200 ms) while it runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
         "pcie.link.gen.current,pcie.link.width.current")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None
        self.pcie = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons, gens, widths = [], [], set(), [], []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        try:
            with open(self.path) as f:
                for line in f:
                    p = [x.strip() for x in line.split(",")]
                    if len(p) < 9:
                        continue
                    try:
                        sm.append(float(p[1]))
                        mx.append(float(p[2]))
                    except ValueError:
                        continue
                    for n, v in zip(names, p[5:9]):
                        if v.lower() == "active":
                            reasons.add(n)
                    if len(p) >= 11:
                        try:
                            gens.append(int(p[9]))
                            widths.append(int(p[10]))
                        except ValueError:
                            pass
            os.unlink(self.path)
        except OSError:
            pass
        self.pcie = {"gen": max(gens), "width": max(widths)} if gens else None
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- roofline model

def layer_params(s) -> int:
    H, I = s.hidden, s.inter
    return H * (s.n_q + 2 * s.n_kv) + s.n_q * H + 3 * H * I


def attn_fwd_flop(s, seq_len, nseq) -> float:
    # QK^T and PV over the causal triangle
    return 4.0 * s.heads * s.head_dim * nseq * seq_len * (seq_len + 1) / 2


def pcie_link(gpu_index: int) -> dict:
    """Host link of the GPU as nvidia-smi reports it (read-only query): PCIe generation and
    width now and at most, and the per-direction payload rate that generation x width
    gives (GT/s per lane x lanes x line-code efficiency / 8)."""
    q = "pcie.link.gen.current,pcie.link.gen.max,pcie.link.width.current,pcie.link.width.max"
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={q}", "--format=csv,noheader,nounits"],
                             capture_output=True, text=True, timeout=30).stdout.strip().split(",")
        gen, gen_max, width, width_max = (int(x.strip()) for x in out[:4])
    except (OSError, ValueError, subprocess.TimeoutExpired):
        return {"gen": None, "width": None}
    return {"gen": gen, "gen_max": gen_max, "width": width, "width_max": width_max,
            "spec_gbs_per_direction": round(pcie_spec_gbs(gen_max, width_max), 2)}


def pcie_path(gpu_index: int) -> dict:
    """Every PCIe hop between the GPU and the root port, as sysfs lists them (read-only):
    each device's current link speed (GT/s) and width, and the slowest hop's payload
    rate, which bounds host-to-device copies no matter what the GPU's own link says."""
    try:
        bus = subprocess.run(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=30).stdout.strip()
        dom, rest = bus.split(":", 1)
        bdf = f"{int(dom, 16) & 0xFFFF:04x}:{rest.lower()}"
        path = os.path.realpath(f"/sys/bus/pci/devices/{bdf}")
    except (OSError, ValueError, subprocess.TimeoutExpired):
        return {"hops": None}
    hops = []
    d = path
    while re.fullmatch(r"[0-9a-f]{4}:[0-9a-f]{2}:[0-9a-f]{2}\.[0-7]", os.path.basename(d)):
        try:
            sp = open(os.path.join(d, "current_link_speed")).read().split()[0]
            wd = int(open(os.path.join(d, "current_link_width")).read().strip())
            gts = float(sp)
        except (OSError, ValueError, IndexError):
            gts, wd = None, None
        if gts and wd:
            gen = {2.5: 1, 5.0: 2, 8.0: 3, 16.0: 4, 32.0: 5, 64.0: 6}.get(gts)
            hops.append({"device": os.path.basename(d), "gts": gts, "width": wd, "gen": gen,
                         "gbs": round(pcie_spec_gbs(gen, wd), 2) if gen else None})
        d = os.path.dirname(d)
    rated = [h for h in hops if h["gbs"]]
    slow = min(rated, key=lambda h: h["gbs"]) if rated else None
    return {"hops": hops, "slowest": slow}


def pcie_spec_gbs(gen: int, width: int) -> float:
    """Per-direction payload rate of a PCIe link: Gen1/2 8b/10b, Gen3-5 128b/130b, Gen6
    FLIT mode (242 payload bytes per 256)."""
    gts = {1: 2.5, 2: 5.0, 3: 8.0, 4: 16.0, 5: 32.0, 6: 64.0}.get(gen)
    if gts is None:
        return float("nan")
    eff = 0.8 if gen <= 2 else (128 / 130 if gen <= 5 else 242 / 256)
    return gts * width * eff / 8


def link_roofline_ms(s, T, seq_len, nseq, stats_k, layer_bytes, vocab_chunk_bytes, nvch, tflops, link_gbs,
                     shared_read) -> dict:
    """The per-read roofline of one step from the reads the schedule actually made: every
    use of a layer or vocabulary chunk costs max(its FLOPs / tensor peak, its bytes / link)
    when it was copied, and its FLOPs alone when a slot still held it (a reuse).  Reused
    items are charged the smaller (forward) compute, so this never overstates the bound.
    Uses per step: layers 2L (shared-read DPO, SFT) or 3L (two forward sweeps), chunks
    likewise."""
    P = layer_params(s)
    r = s.lora_r
    lora_f = 2.0 * T * r * (2 * s.hidden + s.n_q + s.n_kv)
    att = attn_fwd_flop(s, seq_len, nseq)
    needs_ref = s.method in ("dpo", "kto")
    rows = 2 * T if needs_ref and shared_read else T
    f_fwd = 2.0 * rows * P + att * rows / T + lora_f
    f_bwd = 2.0 * T * P + 2 * att + 2 * lora_f
    vrows = math.ceil(s.vocab / nvch)
    fv_fwd = 2.0 * rows * vrows * s.hidden
    fv_bwd = 2.0 * T * vrows * s.hidden   # dH; the logits recomputed for the softmax are not counted
    n_fwd_sweeps = 2 if needs_ref and not shared_read else 1
    if n_fwd_sweeps == 2:
        f_fwd = 2.0 * T * P + att + lora_f / 2
        fv_fwd = 2.0 * T * vrows * s.hidden
    uses_l = (n_fwd_sweeps + 1) * s.layers
    uses_v = (n_fwd_sweeps + 1) * nvch
    reads_l, reads_v = stats_k["layer_reads"], stats_k["vocab_reads"]
    pk, bw = tflops * 1e12, link_gbs * 1e9
    t = (n_fwd_sweeps * s.layers * max(f_fwd / pk, layer_bytes / bw) + s.layers * max(f_bwd / pk, layer_bytes / bw)
         + n_fwd_sweeps * nvch * max(fv_fwd / pk, vocab_chunk_bytes / bw) + nvch * max(fv_bwd / pk, vocab_chunk_bytes / bw))
    # a reuse saves the copy of the cheaper use of that item
    t -= max(0.0, uses_l - reads_l) * (max(f_fwd / pk, layer_bytes / bw) - f_fwd / pk)
    t -= max(0.0, uses_v - reads_v) * (max(fv_fwd / pk, vocab_chunk_bytes / bw) - fv_fwd / pk)
    flop = (n_fwd_sweeps * s.layers * f_fwd + s.layers * f_bwd + n_fwd_sweeps * nvch * fv_fwd + nvch * fv_bwd)
    return {"ms": t * 1e3, "flop": flop, "link_ms": stats_k["h2d_bytes"] / bw * 1e3,
            "compute_ms": flop / pk * 1e3}


def h2d_peak_gbs(dev, nbytes=1 << 30, reps=5) -> float:
    """Best pinned-host -> device copy rate of one large cudaMemcpyAsync."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(dev)
    best = 0.0
    with torch.cuda.stream(s):
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            d.copy_(h, non_blocking=True)
            e1.record(s)
            s.synchronize()
            best = max(best, nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del h, d
    return best


# ----------------------------------------------------------------------------- CPU oracle sample

def oracle_sample(s, seed: int, layer: int, T_tokens, cu, mask, prep=None):
    """Time 1/L of one step of the oracle: one decoder layer (policy forward with the
    adapter + backward, reference forward without it) and 1/L of the vocabulary head
    (logits, log-sum-exp, target logprob, backward to the hidden state)."""
    from oracle import model as om
    if prep is None or prep.get("layer") != layer:
        w = {n: om.dequant_weight(synth.weight(s, layer, n, seed)) for n in ("q", "k", "v", "o", "gate", "up", "down")}
        lw = om.LayerWeights(w["q"], w["k"], w["v"], w["o"], w["gate"], w["up"], w["down"],
                             om.t64(synth.norm_weight(s, layer, 0, seed)), om.t64(synth.norm_weight(s, layer, 1, seed)))
        aq, bq = synth.lora_weights(s, layer, "q", seed)
        av, bv = synth.lora_weights(s, layer, "v", seed)
        ad = om.Adapter(om.t64(aq), om.t64(bq), om.t64(av), om.t64(bv))
        rows = (s.vocab + s.layers - 1) // s.layers
        head = om.dequant_weight(synth.weight(s, -1, "lm_head", seed, row0=0, nrows=rows))
        x = om.t64(synth.gaussian((len(T_tokens), s.hidden), seed, 900, layer))
        prep = {"layer": layer, "lw": lw, "ad": ad, "head": head, "x": x}
    lw, ad, head, x = prep["lw"], prep["ad"], prep["head"], prep["x"]
    t0 = time.perf_counter()
    for p in ad.params():
        p.requires_grad_(True)
        p.grad = None
    xin = x.clone().requires_grad_(True)
    y = om.decoder_layer(xin, lw, ad, s, cu, adapter_on=True)
    if s.method in ("dpo", "kto"):
        with torch.no_grad():
            om.decoder_layer(x, lw, ad, s, cu, adapter_on=False)
    hf = x.clone().requires_grad_(True)
    logits = hf @ head.T
    lse = torch.logsumexp(logits, dim=-1)
    if s.method in ("dpo", "kto"):
        with torch.no_grad():
            torch.logsumexp(x @ head.T, dim=-1)
    (y.sum() * 1e-3 + lse.sum() * 1e-3).backward()
    dt = time.perf_counter() - t0
    return dt, prep


def run_oracle_arm(args, s, ws, rank):
    tok, cu, mask = synth.tokens(s), synth.seq_offsets(s), synth.loss_mask(s)
    cores = torch.get_num_threads()
    prep = None
    for _ in range(args.warmup):
        _, prep = oracle_sample(s, 0, 0, tok, cu, mask, prep)
    times = []
    for _ in range(args.steps):
        dt, prep = oracle_sample(s, 0, 0, tok, cu, mask, prep)
        times.append(dt)
    # one timed step is the sample, 1/L of the training step: it advances T / L tokens
    sample_s = sum(times) / len(times)
    return s.tokens / s.layers / sample_s, sample_s, cores


# ----------------------------------------------------------------------------- GPU arm

def timed_steps(st, step, steps: int, dev, ws: int, clk=None):
    """K steps on the stack's compute stream between CUDA events, barrier and device
    synchronisation on both sides; returns (max over ranks of the ms, stats of the K steps)."""
    st.stats(reset=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize(dev)
    e0.record(st.compute)
    for _ in range(steps):
        step()
    e1.record(st.compute)
    torch.cuda.synchronize(dev)
    barrier(ws)
    stats = st.stats(reset=True)
    return max_over_ranks(e0.elapsed_time(e1), ws, dev), stats


def per_step(stats, K):
    return {k: stats[k] / K for k in ("layer_reads", "vocab_reads", "h2d_bytes", "kernel_launches", "slot_reuses")}


def make_step(L, st, s, tok, cu, mask, count, flat, holder):
    """One training step as the library runs it: forward(s), loss, streamed backward,
    gradient gather, AdamW on the adapters."""
    def step():
        if s.method == "sft":
            holder["out"] = st.sft_step(tok, cu, mask, count, holder.get("out"))
        else:
            holder["out"] = st.pref_step(s.method, tok, cu, mask, holder.get("out"))
        L.check(L.lib().lora_grads(st.ctx, flat.data_ptr(), 0), st.ctx)
        st.optimizer_step(zero_grads=True)
    return step


def roof_for(L, st, s, stats_k, tf_peak, link):
    layer_img = L.layer_layout(st.cfg)[1]
    nvch = st.stats()["vocab_chunks"]
    return link_roofline_ms(s, s.tokens, s.seq_len, s.nseq, stats_k, layer_img, s.vocab * s.hidden * NF4_BYTES_PER_PARAM / nvch,
                            nvch, tf_peak, link, st.shared_read)


def run_sft_leg(L, args, s, base, dev, ws, tf_peak, link):
    """The SFT step at the same shape and batch (every position of both sequences is a
    target), on the same pinned base: tokens/s, layer reads, peak device bytes."""
    s = s.with_(method="sft", prompt_len=0)
    torch.cuda.empty_cache()
    torch.cuda.reset_peak_memory_stats(dev)
    mem0 = torch.cuda.memory_allocated(dev)
    st = L.Stack(s, device=str(dev))
    st.adopt_base(base)
    st.set_adapters_synthetic(synth, seed=0)
    tok_np, cu_np, mask_np = synth.tokens(s, 0), synth.seq_offsets(s), synth.loss_mask(s)
    tok, cu, mask = st.upload_batch(tok_np, cu_np, mask_np)
    flat = torch.empty(st.grad_numel(), dtype=torch.float32, device=dev)
    st.init_optimizer(lr=1e-4)
    holder = {}
    step = make_step(L, st, s, tok, cu, mask, float(mask_np.sum()), flat, holder)
    for _ in range(args.warmup):
        step()
    if st.sync(600000) != 0:
        raise RuntimeError(L.last_error(st.ctx))
    K = args.steps
    ms, stats = timed_steps(st, step, K, dev, ws)
    if st.sync(60000) != 0:
        raise RuntimeError(L.last_error(st.ctx))
    peak = torch.cuda.max_memory_allocated(dev) - mem0
    sk = per_step(stats, K)
    roof = roof_for(L, st, s, sk, tf_peak, link)
    out = {"workload": f"{s.name} streamed NF4 LoRA SFT, {s.nseq} x {s.seq_len} tokens", "value": round(ws * s.tokens * K / (ms * 1e-3), 2),
           "unit": UNIT, "ms_per_step": round(ms / K, 3), "layer_reads_per_step": sk["layer_reads"],
           "vocab_chunk_reads_per_step": sk["vocab_reads"], "h2d_gb_per_step": round(sk["h2d_bytes"] / 1e9, 3),
           "h2d_gbs": round(sk["h2d_bytes"] / (ms / K * 1e-3) / 1e9, 2),
           "step_roofline_ms": round(roof["ms"], 3), "step_roofline_frac": round(roof["ms"] / (ms / K), 4),
           "workspace_bytes": int(st.ws_bytes), "peak_device_bytes": int(peak),
           "loss": float(holder["out"]["loss"].item())}
    st.close()
    del st
    torch.cuda.empty_cache()
    return out


def run_gpu_arm(args, s, ws, rank, local):
    import layer_streamed_nf4_dequant_b300 as L

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    peaks = read_peaks()
    link = h2d_peak_gbs(dev)
    pcie = pcie_link(local)
    pcie["path"] = pcie_path(local)
    tf_peak = peaks["bf16_tflops_sustained"]

    torch.cuda.empty_cache()
    torch.cuda.reset_peak_memory_stats(dev)
    mem0 = torch.cuda.memory_allocated(dev)
    t_load = time.perf_counter()
    st = L.Stack(s, device=str(dev))
    st.load_synthetic(synth, seed=0)
    st.set_adapters_synthetic(synth, seed=0)
    layer_file = None
    if args.stream_source == "file":
        # the NVMe tier: layer images in a file, read through pinned staging buffers
        layer_file = os.path.join(args.file_dir or tempfile.gettempdir(), f"ls_layers_{os.getpid()}_{rank}.bin")
        st.write_layer_file(layer_file)
        st.use_layer_file(layer_file, nbuf=args.stage_buffers)
    t_load = time.perf_counter() - t_load
    data_seed = rank  # weak scaling: each replica trains on its own pair
    tok_np, cu_np, mask_np = synth.tokens(s, data_seed), synth.seq_offsets(s), synth.loss_mask(s)
    tok, cu, mask = st.upload_batch(tok_np, cu_np, mask_np)
    flat = torch.empty(st.grad_numel(), dtype=torch.float32, device=dev)
    st.init_optimizer(lr=1e-4)
    holder = {}
    step = make_step(L, st, s, tok, cu, mask, float(mask_np.sum()), flat, holder)

    step()
    if st.sync(600000) != 0:
        raise RuntimeError(L.last_error(st.ctx))
    loss_first = float(holder["out"]["loss"].item())   # the optimizer then keeps training on this one batch
    for _ in range(args.warmup - 1):
        step()
    if st.sync(600000) != 0:
        raise RuntimeError(L.last_error(st.ctx))
    torch.cuda.synchronize(dev)

    # ---------------- timed region: batch resident on the device
    K = args.steps
    with ClockSampler(local) as clk:
        ms_max, stats = timed_steps(st, step, K, dev, ws)
    if st.sync(60000) != 0:
        raise RuntimeError(L.last_error(st.ctx))
    loss = float(holder["out"]["loss"].item())
    peak_dev = torch.cuda.max_memory_allocated(dev) - mem0

    # ---------------- the same steps again, every kernel bracketed by CUDA events on the
    # compute stream (per-kernel durations for the roofline; the events slow the step a
    # little, so the throughput above is taken without them); the loss of each step is
    # read back here, outside the timed region
    L.check(L.lib().ls_profile(st.ctx, 1), st.ctx)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    losses = torch.empty(K, dtype=torch.float32, device=dev)
    p0.record(st.compute)
    for i in range(K):
        step()
        with torch.cuda.stream(st.compute):
            losses[i].copy_(holder["out"]["loss"][0])
    p1.record(st.compute)
    torch.cuda.synchronize(dev)
    prof_step_ms = p0.elapsed_time(p1) / K
    prof = L.ls_profile_t()
    L.check(L.lib().ls_profile_read(st.ctx, prof), st.ctx)
    L.check(L.lib().ls_profile(st.ctx, 0), st.ctx)
    st.stats(reset=True)
    loss_traj = [float(x) for x in losses.cpu()]

    # ---------------- e2e: pinned host batch in, loss out, every step
    h_tok = torch.from_numpy(tok_np).pin_memory()
    h_cu = torch.from_numpy(cu_np).pin_memory()
    h_mask = torch.from_numpy(mask_np).pin_memory()
    h_loss = torch.empty(1, dtype=torch.float32, pin_memory=True)
    bufs = {}
    for _ in range(2):
        st.train_step(h_tok, h_cu, h_mask, s.method, s.beta, h_loss, flat, bufs)
    barrier(ws)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(K):
        st.train_step(h_tok, h_cu, h_mask, s.method, s.beta, h_loss, flat, bufs)
    torch.cuda.synchronize(dev)
    e2e_s = time.perf_counter() - t0
    barrier(ws)
    e2e_max = max_over_ranks(e2e_s, ws, dev)
    st.stats(reset=True)

    step_ms = ms_max / K
    tokens_per_step = s.tokens
    value = ws * tokens_per_step * K / (ms_max * 1e-3)
    e2e_value = ws * tokens_per_step * K / e2e_max

    p = prof.as_dict()
    dom = max(("gemm_fwd", "gemm_dx"), key=lambda k: p[k]["ms"])
    achieved = p[dom]["flop"] / (p[dom]["ms"] * 1e-3) / 1e12 if p[dom]["ms"] > 0 else 0.0
    total_prof_ms = sum(v["ms"] for v in p.values())

    stats_k = per_step(stats, K)
    roof = roof_for(L, st, s, stats_k, tf_peak, link)
    clocks = clk.summary()
    file_stats = None
    if args.stream_source == "file":
        file_stats = {"file_gb_per_step": round(stats["file_bytes"] / K / 1e9, 3),
                      "file_read_gbs": round(stats["file_bytes"] / max(1e-9, stats["file_read_ms"] * 1e-3) / 1e9, 2),
                      "file_seq_read_gbs": round(file_read_peak_gbs(layer_file, st.layer_file_stride()), 2),
                      "staging_buffers": args.stage_buffers}
    workspace = int(st.ws_bytes)
    shared = bool(st.shared_read)

    # ---------------- SFT at the same shape and batch (the metric's "SFT+DPO")
    sft = None
    if s.method != "sft" and not args.no_sft and args.stream_source == "ram":
        sft = run_sft_leg(L, args, s, st, dev, ws, tf_peak, link)
        sft["dpo_over_sft"] = {"layer_reads": round(stats_k["layer_reads"] / max(1e-9, sft["layer_reads_per_step"]), 4),
                               "peak_device_bytes": round(peak_dev / max(1, sft["peak_device_bytes"]), 4),
                               "pages_layer_reads": 1.52, "pages_peak_memory": 0.914}
    if layer_file:
        try:
            os.unlink(layer_file)
        except OSError:
            pass
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{s.name} streamed NF4 LoRA {s.method.upper()}"
                               + (" (layers from file)" if args.stream_source == "file" else ""), "layers": s.layers,
                   "hidden": s.hidden, "heads": s.heads, "kv_heads": s.kv_heads, "inter": s.inter,
                   "vocab": s.vocab, "lora_r": s.lora_r, "tokens_per_pass": s.tokens,
                   "seqs": s.nseq, "seq_len": s.seq_len, "prompt_len": s.prompt_len,
                   "global_batch_tokens": ws * tokens_per_step, "parallelism": f"replicas x{ws}",
                   "dpo_shared_read": shared,
                   "l2": "inputs larger than L2: each step streams the NF4 base (GBs) from pinned host"},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT,
                "h2d_bytes_per_step": int(h_tok.numel() * 4 + h_cu.numel() * 4 + h_mask.numel()),
                "d2h_bytes_per_step": 4},
        "gpu_launches": int(stats_k["kernel_launches"] * K),
        "roofline": {"bound": "tensor", "kernel": f"nf4_gemm ({dom})", "achieved": round(achieved, 2),
                     "peak": tf_peak, "unit": "TFLOP/s", "frac": round(achieved / tf_peak, 4),
                     "peak_source": f"{peaks['source']} bf16 sustained",
                     "traffic": (round(p[dom]["bytes"] / max(1, p[dom]["launches"]) * GEMM_TRAFFIC_PER_ALG_BYTE[dom])
                                 if GEMM_TRAFFIC_PER_ALG_BYTE.get(dom) else None),
                     "traffic_unit": "bytes per launch (ncu-measured DRAM/algorithmic ratio x algorithmic bytes)",
                     "alg_bytes_per_launch": round(p[dom]["bytes"] / max(1, p[dom]["launches"])),
                     "launches": p[dom]["launches"], "avg_launch_us": round(1e3 * p[dom]["ms"] / max(1, p[dom]["launches"]), 2)},
        "stream": {"h2d_gbs": round(stats_k["h2d_bytes"] / (step_ms * 1e-3) / 1e9, 2),
                   "h2d_peak_gbs": round(link, 2), "h2d_frac_of_peak": round(stats_k["h2d_bytes"] / (step_ms * 1e-3) / 1e9 / link, 4),
                   "pcie": {**pcie, "gen_under_load": (clk.pcie or {}).get("gen"),
                            "width_under_load": (clk.pcie or {}).get("width")},
                   "h2d_gb_per_step": round(stats_k["h2d_bytes"] / 1e9, 3),
                   "layer_reads_per_step": stats_k["layer_reads"], "vocab_chunk_reads_per_step": stats_k["vocab_reads"],
                   "slot_reuses_per_step": stats_k["slot_reuses"],
                   "step_roofline_ms": round(roof["ms"], 3), "step_roofline_frac": round(roof["ms"] / step_ms, 4),
                   "link_ms": round(roof["link_ms"], 3), "compute_at_peak_ms": round(roof["compute_ms"], 3),
                   "step_algorithmic_tflop": round(roof["flop"] / 1e12, 3),
                   "workspace_bytes": workspace, "peak_device_bytes": int(peak_dev),
                   "load_s": round(t_load, 1), "source": args.stream_source,
                   **(file_stats or {})},
        "sft": sft,
        "profiled_ms_per_step": round(prof_step_ms, 3),
        "kernels_ms_per_step": {k: round(v["ms"] / K, 3) for k, v in p.items()},
        "kernels_share": {k: round(v["ms"] / total_prof_ms, 4) for k, v in p.items()} if total_prof_ms else {},
        "loss_first_step": loss_first, "loss": loss, "loss_per_profiled_step": loss_traj,
        "clocks": clocks,
    }
    st.close()
    return res


def file_read_peak_gbs(path: str, stride: int, reps: int = 2) -> float:
    """Plain sequential read rate of the layer file (O_DIRECT where the file system allows
    it, 64 MiB requests into an aligned buffer): the disk tier's bound."""
    import mmap
    size = os.path.getsize(path)
    flags = os.O_RDONLY | getattr(os, "O_DIRECT", 0)
    try:
        fd = os.open(path, flags)
    except OSError:
        fd = os.open(path, os.O_RDONLY)
    buf = mmap.mmap(-1, 64 << 20)
    best = 0.0
    try:
        for _ in range(reps):
            off = 0
            t0 = time.perf_counter()
            while off < size:
                n = os.preadv(fd, [buf], off)
                if n <= 0:
                    break
                off += n
            best = max(best, off / (time.perf_counter() - t0) / 1e9)
    finally:
        os.close(fd)
        buf.close()
    return best


def gemm_microbench(spec: str, reps: int = 10) -> dict:
    """One NF4-dequant-fused matrix product through the C ABI (lsk_nf4_gemm_sk, the
    schedule the training step uses), timed with CUDA events after warm-up:
    spec = "mode,M,N,K[,bn,nacc[,split[,pair_rows]]]" (mode 0: Y = X deq(W)^T, mode 1:
    dX = dY deq(W); W [N, K] drawn N(0, 0.02) and NF4-quantised on the host; split 0 = cost
    model, 1 = split tiles, -1 = whole tiles; pair_rows = M / 2 runs the shared-read
    forward's paired halves)."""
    import layer_streamed_nf4_dequant_b300 as L
    f = [int(x) for x in spec.split(",")]
    mode, M, N, K = f[:4]
    bn, nacc = (f[4], f[5]) if len(f) >= 6 else (0, 0)
    split = f[6] if len(f) >= 7 else 0
    pair = f[7] if len(f) >= 8 else 0
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(0)
    pk, am = L.quantize_host((torch.randn(N, K, generator=g) * 0.02).numpy())
    p, a = torch.from_numpy(pk).to(dev), torch.from_numpy(am).to(dev)
    red, outc = (K, N) if mode == 0 else (N, K)
    x = torch.randn(M, red, device=dev).to(torch.bfloat16)
    out = torch.empty(M, outc, device=dev, dtype=torch.bfloat16 if mode == 0 else torch.float32)
    st = torch.cuda.current_stream().cuda_stream
    ws = torch.zeros(int(L.lib().lsk_nf4_gemm_workspace_bytes()), dtype=torch.uint8, device=dev)

    def run():
        L.call("lsk_nf4_gemm_sk", mode, x, red, M, p, a, N, K, None, None, 0, 0 if mode == 0 else 1, out, outc, None,
               0, bn, nacc, split, pair, ws, ws.numel(), st)

    for _ in range(3):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        run()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / reps * 1e3
    peaks = read_peaks()
    tf = 2.0 * M * N * K / (us * 1e-6) / 1e12
    return {"kernel": "nf4_gemm", "mode": mode, "M": M, "N": N, "K": K, "bn": bn, "nacc": nacc, "split": split,
            "pair_rows": pair,
            "us": round(us, 2), "tflops": round(tf, 1), "frac_of_burst_peak": round(tf / peaks["bf16_tflops"], 4),
            "peak_source": peaks["source"]}


def attn_microbench(spec: str, reps: int = 10) -> dict:
    """Causal GQA attention forward and backward through the C ABI (lsk_attn_fwd /
    lsk_attn_bwd, the tcgen05 kernels the training step runs), timed with CUDA events after
    warm-up: spec = "T,nseq,nh,nkv,hd" (nseq equal sequences of T / nseq tokens; q/k/v and dO
    drawn N(0, 1) in bf16; the backward takes the per-query-head split the step uses when
    nh > nkv).  FLOPs: forward 4 hd nh sum L(L+1)/2, backward 2.5x that."""
    import layer_streamed_nf4_dequant_b300 as L
    T, nseq, nh, nkv, hd = [int(x) for x in spec.split(",")]
    if nseq < 1 or T % nseq or nh % nkv:
        raise ValueError("attn spec: T,nseq,nh,nkv,hd with T a multiple of nseq and nh of nkv")
    Ls = T // nseq
    cu = list(range(0, T + 1, Ls))
    dev = torch.device("cuda:0")
    ncols = (nh + 2 * nkv) * hd
    g = torch.Generator().manual_seed(0)
    qkv = torch.randn(T, ncols, generator=g).to(torch.bfloat16).to(dev)
    dout = torch.randn(T, nh * hd, generator=g).to(torch.bfloat16).to(dev)
    cud = torch.tensor(cu, dtype=torch.int32, device=dev)
    o = torch.empty((T, nh * hd), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((nh, T), dtype=torch.float32, device=dev)
    dsc = torch.empty((nh, T), dtype=torch.float32, device=dev)
    dq = torch.zeros((T, ncols), dtype=torch.float32, device=dev)
    part = torch.empty((nh // nkv) * T * 2 * nkv * hd, dtype=torch.float32, device=dev) if nh > nkv else None
    st = torch.cuda.current_stream().cuda_stream

    def fwd():
        L.call("lsk_attn_fwd", qkv, ncols, cud, nseq, Ls, nh, nkv, hd, o, nh * hd, lse, T, st)

    def bwd():
        L.call("lsk_attn_bwd", qkv, ncols, dout, o, nh * hd, lse, cud, nseq, Ls, nh, nkv, hd, dsc, dq, ncols, T, part,
               st)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps * 1e3

    fus = timed(fwd)
    bus = timed(bwd)
    flop = 4.0 * hd * nh * nseq * Ls * (Ls + 1) / 2
    return {"kernel": "attention", "T": T, "nseq": nseq, "nh": nh, "nkv": nkv, "hd": hd,
            "fwd_us": round(fus, 2), "fwd_tflops": round(flop / (fus * 1e-6) / 1e12, 1),
            "bwd_us": round(bus, 2), "bwd_tflops": round(2.5 * flop / (bus * 1e-6) / 1e12, 1)}


def cpu_baseline(s, seconds_budget: float = 20.0):
    tok, cu, mask = synth.tokens(s), synth.seq_offsets(s), synth.loss_mask(s)
    _, prep = oracle_sample(s, 0, 0, tok, cu, mask, None)   # warm-up (and weight preparation)
    times = []
    t_start = time.perf_counter()
    while not times or (time.perf_counter() - t_start < seconds_budget and len(times) < 5):
        dt, prep = oracle_sample(s, 0, 0, tok, cu, mask, prep)
        times.append(dt)
    step_s = statistics.median(times) * s.layers
    return {"value": round(s.tokens / step_s, 4), "unit": UNIT, "cores": torch.get_num_threads(), "kind": "oracle",
            "sample": (f"fp64 oracle, 1/{s.layers} of a step ({len(times)} runs): one {s.name} decoder layer at "
                       f"T={s.tokens} (policy fwd+bwd, reference fwd) + {math.ceil(s.vocab / s.layers)} vocabulary rows "
                       f"(fwd, ref fwd, bwd); step time = {s.layers} x median")}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="llama-3.1-8b", choices=sorted(synth.CONFIGS))
    ap.add_argument("--method", default=None, choices=["sft", "dpo", "simpo", "orpo", "kto"],
                    help="training method on the config's pairs (default: the config's own)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gemm", default=None, help="micro-benchmark one NF4 GEMM: mode,M,N,K[,bn,nacc[,split[,pair_rows]]] (split: 0 cost model, 1 split tiles, -1 whole tiles)")
    ap.add_argument("--attn", default=None,
                    help="micro-benchmark causal GQA attention fwd + bwd: T,nseq,nh,nkv,hd (e.g. 1024,2,32,8,128)")
    ap.add_argument("--stream-source", default="ram", choices=["ram", "file"],
                    help="where the streamed decoder layers live: pinned host RAM, or a file (NVMe tier)")
    ap.add_argument("--file-dir", default=None, help="directory of the layer file (default: the temp dir)")
    ap.add_argument("--stage-buffers", type=int, default=3, help="pinned staging buffers of the file tier")
    ap.add_argument("--no-sft", action="store_true", help="skip the SFT leg of a preference-method run")
    ap.add_argument("--layers", type=int, default=0,
                    help="run the config's shape with fewer decoder layers (every kernel keeps its full-size "
                         "shape; for profiling captures, not a bench line)")
    args = ap.parse_args()
    if args.gemm:
        print(json.dumps(gemm_microbench(args.gemm, max(1, args.steps))), flush=True)
        return
    if args.attn:
        print(json.dumps(attn_microbench(args.attn, max(1, args.steps))), flush=True)
        return
    if args.warmup < 3:
        args.warmup = 3
    s = synth.CONFIGS[args.config]
    if args.method and args.method != s.method:
        s = s.with_(method=args.method, prompt_len=0 if args.method == "sft" else s.prompt_len)
    if args.layers:
        s = s.with_(layers=args.layers, name=f"{s.name}-L{args.layers}")
    ws, rank, local = dist_env()

    if args.impl == "reference":
        init_dist(ws, "gloo")
        if rank != 0:
            barrier(ws)
            return
        value, sample_s, cores = run_oracle_arm(args, s, ws, rank)
        line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": ws,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sample_s * 1e3, 1),
                "step": f"1/{s.layers} of a training step ({s.tokens / s.layers:.1f} tokens): one decoder layer + "
                        f"{math.ceil(s.vocab / s.layers)} vocabulary rows; full-step equivalent "
                        f"{sample_s * s.layers:.1f} s",
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": {"workload": f"{s.name} streamed NF4 LoRA {s.method.upper()}", "tokens_per_pass": s.tokens},
                "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                                 "sample": f"each timed step is 1/{s.layers} of a training step (one decoder "
                                           f"layer + {math.ceil(s.vocab / s.layers)} vocabulary rows, "
                                           f"{s.tokens / s.layers:.1f} tokens' worth), timed in full"},
                "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        barrier(ws)
        return

    init_dist(ws, "nccl")
    res = run_gpu_arm(args, s, ws, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline and ws == 1:
            res["cpu_baseline"] = cpu_baseline(s)
        else:
            res["cpu_baseline"] = None
        print(json.dumps(res), flush=True)
    barrier(ws)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
