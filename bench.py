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
run of the same steps with every kernel bracketed by CUDA events.

--impl reference times the CPU oracle (fp64) on a bounded sample of the same
workload: one decoder layer (policy forward + backward, reference forward) plus
1/L of the vocabulary head, i.e. 1/L of a step, scaled by L.
"""
from __future__ import annotations

import argparse
import json
import math
import os
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
# DRAM bytes (read + write) per algorithmic byte of the forward NF4 GEMM, from one ncu
# capture of the 8B gate|up launch on the split schedule (M 2048, N 28672, K 4096:
# 86.0 MB read + 106.1 MB written against 200.3 MB algorithmic; output rows partly still
# in L2 at kernel end).  It scales the class's algorithmic bytes per launch to the
# reported traffic; set to None whenever the kernel changes until it is captured again.
GEMM_FWD_TRAFFIC_PER_ALG_BYTE = 192.1 / 200.3
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
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

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
        sm, mx, reasons = [], [], set()
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
            os.unlink(self.path)
        except OSError:
            pass
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


def step_roofline_ms(s, stats, T, nseq, seq_len, method, tflops, link_gbs, shared_read=False) -> dict:
    """Sum over the step's layer and vocabulary reads of max(FLOPs / tensor peak, bytes / link).

    FLOPs are algorithmic: forward 2 T P + attention; backward 2 T P (the frozen base
    needs input gradients only) + twice the attention forward; LoRA adds 2 T r (K + N)
    per adapted projection and direction.  The backward's recompute is not counted.
    DPO reads every layer once for the policy and once for the reference forward, or
    once for both when they share a sweep (shared_read), then once for the backward.
    """
    P = layer_params(s)
    r = s.lora_r
    lora_f = 2.0 * T * r * (2 * s.hidden + s.n_q + s.n_kv)
    att = attn_fwd_flop(s, seq_len, nseq)
    f_fwd = 2.0 * T * P + att
    f_bwd = 2.0 * T * P + 2 * att + 2 * lora_f
    layer_b = stats["slot_bytes_layer"]
    V, H = s.vocab, s.hidden
    vocab_fwd = 2.0 * T * V * H
    vocab_b = V * H * NF4_BYTES_PER_PARAM
    needs_ref = method in ("dpo", "kto")
    sweeps_fwd = [True, False] if needs_ref else [True]
    t = 0.0
    pk = tflops * 1e12
    bw = link_gbs * 1e9
    if needs_ref and shared_read:
        t += s.layers * max((2 * f_fwd + lora_f) / pk, layer_b / bw)
        t += max(2 * vocab_fwd / pk, vocab_b / bw)
    else:
        for on in sweeps_fwd:
            t += s.layers * max((f_fwd + (lora_f if on else 0.0)) / pk, layer_b / bw)
            t += max(vocab_fwd / pk, vocab_b / bw)
    t += s.layers * max(f_bwd / pk, layer_b / bw)
    t += max(2 * vocab_fwd / pk, vocab_b / bw)   # recomputed logits are not counted; dH is
    return {"ms": t * 1e3, "flop": (len(sweeps_fwd) * (s.layers * f_fwd + vocab_fwd) + s.layers * (f_bwd + lora_f)
                                    + 2 * vocab_fwd)}


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
        times.append(dt * s.layers)   # the sample is 1/L of a step
    step_s = sum(times) / len(times)
    tokens = s.tokens
    return tokens / step_s, step_s, cores


# ----------------------------------------------------------------------------- GPU arm

def run_gpu_arm(args, s, ws, rank, local):
    import layer_streamed_nf4_dequant_b300 as L

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    peaks = read_peaks()
    link = h2d_peak_gbs(dev)

    t_load = time.perf_counter()
    st = L.Stack(s, device=str(dev))
    st.load_synthetic(synth, seed=0)
    st.set_adapters_synthetic(synth, seed=0)
    layer_file = None
    if args.stream_source == "file":
        # the NVMe tier: layer images in a file, read through pinned staging buffers
        layer_file = os.path.join(args.file_dir or tempfile.gettempdir(), f"ls_layers_{os.getpid()}_{rank}.bin")
        st.write_layer_file(layer_file)
        st.use_layer_file(layer_file, nbuf=3)
    t_load = time.perf_counter() - t_load
    data_seed = rank  # weak scaling: each replica trains on its own pair
    tok_np, cu_np, mask_np = synth.tokens(s, data_seed), synth.seq_offsets(s), synth.loss_mask(s)
    tok, cu, mask = st.upload_batch(tok_np, cu_np, mask_np)
    flat = torch.empty(st.grad_numel(), dtype=torch.float32, device=dev)
    out = None

    st.init_optimizer(lr=1e-4)

    def step():
        nonlocal out
        if s.method == "sft":
            out = st.sft_step(tok, cu, mask, float(mask_np.sum()), out)
        else:
            out = st.pref_step(s.method, tok, cu, mask, out)
        L.check(L.lib().lora_grads(st.ctx, flat.data_ptr(), 0), st.ctx)
        st.optimizer_step(zero_grads=True)

    step()
    if st.sync(600000) != 0:
        raise RuntimeError(L.last_error(st.ctx))
    loss_first = float(out["loss"].item())   # the optimizer then keeps training on this one batch
    for _ in range(args.warmup - 1):
        step()
    if st.sync(600000) != 0:
        raise RuntimeError(L.last_error(st.ctx))
    torch.cuda.synchronize(dev)

    # ---------------- timed region: batch resident on the device
    st.stats(reset=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        e0.record(st.compute)
        for _ in range(args.steps):
            step()
        e1.record(st.compute)
        torch.cuda.synchronize(dev)
    barrier(ws)
    ms_dev = e0.elapsed_time(e1)
    stats = st.stats(reset=True)
    if st.sync(60000) != 0:
        raise RuntimeError(L.last_error(st.ctx))
    loss = float(out["loss"].item())
    ms_max = max_over_ranks(ms_dev, ws, dev)

    # ---------------- the same steps again, every kernel bracketed by CUDA events on the
    # compute stream (per-kernel durations for the roofline; the events slow the step a
    # little, so the throughput above is taken without them)
    L.check(L.lib().ls_profile(st.ctx, 1), st.ctx)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(st.compute)
    for _ in range(args.steps):
        step()
    p1.record(st.compute)
    torch.cuda.synchronize(dev)
    prof_step_ms = p0.elapsed_time(p1) / args.steps
    prof = L.ls_profile_t()
    L.check(L.lib().ls_profile_read(st.ctx, prof), st.ctx)
    L.check(L.lib().ls_profile(st.ctx, 0), st.ctx)
    st.stats(reset=True)

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
    for _ in range(args.steps):
        st.train_step(h_tok, h_cu, h_mask, s.method, s.beta, h_loss, flat, bufs)
    torch.cuda.synchronize(dev)
    e2e_s = time.perf_counter() - t0
    barrier(ws)
    e2e_max = max_over_ranks(e2e_s, ws, dev)
    st.stats(reset=True)

    K = args.steps
    step_ms = ms_max / K
    tokens_per_step = s.tokens
    value = ws * tokens_per_step * K / (ms_max * 1e-3)
    e2e_value = ws * tokens_per_step * K / e2e_max

    p = prof.as_dict()
    dom = max(("gemm_fwd", "gemm_dx"), key=lambda k: p[k]["ms"])
    tf_peak = peaks["bf16_tflops_sustained"]
    achieved = p[dom]["flop"] / (p[dom]["ms"] * 1e-3) / 1e12 if p[dom]["ms"] > 0 else 0.0
    total_prof_ms = sum(v["ms"] for v in p.values())

    layer_img = L.layer_layout(st.cfg)[1]
    stats_k = {k: v / K for k, v in stats.items() if k in ("layer_reads", "vocab_reads", "h2d_bytes",
                                                            "kernel_launches", "slot_reuses")}
    roof = step_roofline_ms(s, {"slot_bytes_layer": layer_img}, s.tokens, s.nseq, s.seq_len, s.method,
                            tf_peak, link, st.shared_read)
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
                   "dpo_shared_read": bool(st.shared_read),
                   "l2": "inputs larger than L2: each step streams the NF4 base (GBs) from pinned host"},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT,
                "h2d_bytes_per_step": int(h_tok.numel() * 4 + h_cu.numel() * 4 + h_mask.numel()),
                "d2h_bytes_per_step": 4},
        "gpu_launches": int(stats_k["kernel_launches"] * K),
        "roofline": {"bound": "tensor", "kernel": f"nf4_gemm ({dom})", "achieved": round(achieved, 2),
                     "peak": tf_peak, "unit": "TFLOP/s", "frac": round(achieved / tf_peak, 4),
                     "peak_source": f"{peaks['source']} bf16 sustained",
                     "traffic": (round(p[dom]["bytes"] / max(1, p[dom]["launches"]) * GEMM_FWD_TRAFFIC_PER_ALG_BYTE)
                                 if dom == "gemm_fwd" and GEMM_FWD_TRAFFIC_PER_ALG_BYTE else None),
                     "traffic_unit": "bytes per launch (ncu-measured DRAM/algorithmic ratio x algorithmic bytes)",
                     "alg_bytes_per_launch": round(p[dom]["bytes"] / max(1, p[dom]["launches"])),
                     "launches": p[dom]["launches"], "avg_launch_us": round(1e3 * p[dom]["ms"] / max(1, p[dom]["launches"]), 2)},
        "stream": {"h2d_gbs": round(stats_k["h2d_bytes"] / (step_ms * 1e-3) / 1e9, 2),
                   "h2d_peak_gbs": round(link, 2), "h2d_gb_per_step": round(stats_k["h2d_bytes"] / 1e9, 3),
                   "layer_reads_per_step": stats_k["layer_reads"], "vocab_chunk_reads_per_step": stats_k["vocab_reads"],
                   "slot_reuses_per_step": stats_k["slot_reuses"],
                   "step_roofline_ms": round(roof["ms"], 3), "step_roofline_frac": round(roof["ms"] / step_ms, 4),
                   "step_algorithmic_tflop": round(roof["flop"] / 1e12, 3),
                   "workspace_bytes": int(st.ws_bytes), "peak_device_bytes": int(torch.cuda.max_memory_allocated(dev)),
                   "load_s": round(t_load, 1), "source": args.stream_source,
                   **({"file_gb_per_step": round(stats["file_bytes"] / K / 1e9, 3),
                       "file_read_gbs": round(stats["file_bytes"] / max(1e-9, stats["file_read_ms"] * 1e-3) / 1e9, 2)}
                      if args.stream_source == "file" else {})},
        "profiled_ms_per_step": round(prof_step_ms, 3),
        "kernels_ms_per_step": {k: round(v["ms"] / K, 3) for k, v in p.items()},
        "kernels_share": {k: round(v["ms"] / total_prof_ms, 4) for k, v in p.items()} if total_prof_ms else {},
        "loss_first_step": loss_first, "loss": loss,
        "clocks": clk.summary(),
    }
    st.close()
    return res


def gemm_microbench(spec: str, reps: int = 10) -> dict:
    """One NF4-dequant-fused matrix product through the C ABI (lsk_nf4_gemm_sk, the
    schedule the training step uses), timed with CUDA events after warm-up:
    spec = "mode,M,N,K[,bn,nacc[,split]]" (mode 0: Y = X deq(W)^T, mode 1: dX = dY deq(W);
    W [N, K] drawn N(0, 0.02) and NF4-quantised on the host; split 0 = cost model,
    1 = split tiles, -1 = whole tiles)."""
    import layer_streamed_nf4_dequant_b300 as L
    f = [int(x) for x in spec.split(",")]
    mode, M, N, K = f[:4]
    bn, nacc = (f[4], f[5]) if len(f) >= 6 else (0, 0)
    split = f[6] if len(f) >= 7 else 0
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
               0, bn, nacc, split, 0, ws, ws.numel(), st)

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
            "us": round(us, 2), "tflops": round(tf, 1), "frac_of_burst_peak": round(tf / peaks["bf16_tflops"], 4),
            "peak_source": peaks["source"]}


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
    ap.add_argument("--gemm", default=None, help="micro-benchmark one NF4 GEMM: mode,M,N,K[,bn,nacc[,split]] (split: 0 cost model, 1 split tiles, -1 whole tiles)")
    ap.add_argument("--stream-source", default="ram", choices=["ram", "file"],
                    help="where the streamed decoder layers live: pinned host RAM, or a file (NVMe tier)")
    ap.add_argument("--file-dir", default=None, help="directory of the layer file (default: the temp dir)")
    args = ap.parse_args()
    if args.gemm:
        print(json.dumps(gemm_microbench(args.gemm, max(1, args.steps))), flush=True)
        return
    if args.warmup < 3:
        args.warmup = 3
    s = synth.CONFIGS[args.config]
    if args.method and args.method != s.method:
        s = s.with_(method=args.method, prompt_len=0 if args.method == "sft" else s.prompt_len)
    ws, rank, local = dist_env()

    if args.impl == "reference":
        init_dist(ws, "gloo")
        if rank != 0:
            barrier(ws)
            return
        value, step_s, cores = run_oracle_arm(args, s, ws, rank)
        line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": ws,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 1),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": {"workload": f"{s.name} streamed NF4 LoRA {s.method.upper()}", "tokens_per_pass": s.tokens},
                "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                                 "sample": f"1/{s.layers} of a step per timed step (one decoder layer + "
                                           f"{math.ceil(s.vocab / s.layers)} vocabulary rows), scaled by {s.layers}"},
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
