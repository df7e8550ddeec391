"""Decoder stack, losses and LoRA gradients — oracle (test infrastructure only).

Plain resident computation in fp64 (torch CPU), one full matrix product per
linear, no streaming, no tiling.  The model is the Llama-style decoder the Soup
pages train with LoRA (any HF AutoModelForCausalLM text model, axbrief.com
"The Architecture of Low-VRAM Alignment"; Llama-3.1-8B and Qwen2.5-3B in "The
Core Idea: Layer Streaming" of Soup: Fine-Tune an 8B Model on a 4 GB GPU):
pre-norm RMSNorm, q/k/v/o projections without biases, rotate-half RoPE, causal
grouped-query attention, SwiGLU MLP, final RMSNorm, vocabulary projection.

LoRA (same page, soup.yaml listing: r = 16 on q_proj and v_proj; "plain-LoRA" in
its caveats): y = x W^T + u B^T with u = bf16(s * x A^T), s = alpha / r, only A
and B train.  SFT is next-token cross-entropy (axbrief.com, "The Architecture of
Low-VRAM Alignment", SFT then preference losses).  DPO's reference logprobs are
the same base run with the adapter switched off (Show HN: Fine-tune an 8B model
on a 4 GB laptop GPU, first paragraph; evermx.com summary), so a reference pass
here is the same forward with adapter_on=False.

bf16 storage is emulated (round to nearest even) where the GPU path stores bf16:
layer input/output, normed activations, q/k/v after projection and after RoPE,
attention output, the LoRA down-projection u, gate/up, the SwiGLU product.
Logits, log-sum-exp and logprobs stay fp64.  Readings where the pages are silent:
single rounding of residual sums (x + o W_o^T rounded once), RMSNorm as
bf16(w * bf16(x * rstd)), no RoPE frequency scaling, contiguous GQA groups.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch
import torch.nn.functional as F

from .nf4 import nf4_dequantize, nf4_quantize

F64 = torch.float64


# bf16 storage emulation; False gives the pure-fp64 mode (finite differences, invariants).
ROUND = True


def bf16r(x: torch.Tensor) -> torch.Tensor:
    """Round to bf16 (via fp32, nearest even), gradient passed straight through."""
    if not ROUND:
        return x
    r = x.detach().to(torch.float32).to(torch.bfloat16).to(F64)
    return x + (r - x.detach())


class pure_fp64:
    """Context manager: run the oracle without bf16 storage emulation."""

    def __enter__(self):
        global ROUND
        self._old, ROUND = ROUND, False

    def __exit__(self, *exc):
        global ROUND
        ROUND = self._old


class accumulate_in:
    """Context manager: run the oracle's arithmetic in another floating type (fp32).

    Not a second reference: the computation and its bf16 storage points are the same,
    only the accumulation precision drops.  Tests compare such a run with the fp64 one
    to measure how far rounding alone moves a result (its conditioning floor) -- the
    spread any fp32-accumulating implementation may legitimately show.  Weights and
    adapters must be cast with cast_stack / cast_adapters inside the context.
    """

    def __init__(self, dtype=torch.float32):
        self.dtype = dtype

    def __enter__(self):
        global F64
        self._old, F64 = F64, self.dtype

    def __exit__(self, *exc):
        global F64
        F64 = self._old


def t64(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(F64)


# --------------------------------------------------------------------------- weights

@dataclasses.dataclass
class LayerWeights:
    """Dequantised frozen weights of one decoder layer (fp64 holding bf16 values)."""
    wq: torch.Tensor
    wk: torch.Tensor
    wv: torch.Tensor
    wo: torch.Tensor
    wg: torch.Tensor
    wu: torch.Tensor
    wd: torch.Tensor
    w1: torch.Tensor      # attention RMSNorm weight [H]
    w2: torch.Tensor      # MLP RMSNorm weight [H]


@dataclasses.dataclass
class Adapter:
    """LoRA factors of one layer: A [r, K], B [N, r] for q and v (fp64 leaves)."""
    aq: torch.Tensor
    bq: torch.Tensor
    av: torch.Tensor
    bv: torch.Tensor

    def params(self) -> List[torch.Tensor]:
        return [self.aq, self.bq, self.av, self.bv]


def dequant_weight(w: np.ndarray) -> torch.Tensor:
    """NF4-quantise an fp32 weight and return its dequantised values (fp64)."""
    codes, absmax = nf4_quantize(w)
    return t64(nf4_dequantize(codes, absmax))


# --------------------------------------------------------------------------- blocks

def rmsnorm(x: torch.Tensor, w: torch.Tensor, eps: float) -> torch.Tensor:
    """y = bf16(w * bf16(x * rstd)), rstd = 1 / sqrt(mean(x^2) + eps) per row."""
    rstd = 1.0 / torch.sqrt((x * x).mean(dim=-1, keepdim=True) + eps)
    return bf16r(w * bf16r(x * rstd))


def lora_u(x: torch.Tensor, a: torch.Tensor, s: float) -> torch.Tensor:
    """LoRA down-projection stored in bf16: u = bf16(s * x A^T)."""
    return bf16r(s * (x @ a.T))


def linear(x: torch.Tensor, w: torch.Tensor, lora: Optional[tuple] = None,
           residual: Optional[torch.Tensor] = None) -> torch.Tensor:
    """bf16(residual + x W^T + u B^T): one rounding of the fp64 sum."""
    y = x @ w.T
    if lora is not None:
        u, b = lora
        y = y + u @ b.T
    if residual is not None:
        y = residual + y
    return bf16r(y)


def rope(x: torch.Tensor, pos: torch.Tensor, theta: float) -> torch.Tensor:
    """Rotate-half RoPE on x [T, heads, hd]; pair (i, i + hd/2) turned by pos * theta^(-2i/hd)."""
    hd = x.shape[-1]
    half = hd // 2
    inv = theta ** (-2.0 * torch.arange(half, dtype=F64) / hd)
    ang = pos.to(F64)[:, None] * inv[None, :]
    c, s = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return bf16r(torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=-1))


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu: Sequence[int]) -> torch.Tensor:
    """Causal GQA softmax(q k^T / sqrt(hd)) v per sequence; q [T, nh, hd], k/v [T, kv, hd].

    Query head h reads key/value head floor(h * kv / nh) (contiguous groups).
    """
    T, nh, hd = q.shape
    kv = k.shape[1]
    out = []
    for si in range(len(cu) - 1):
        a, b = int(cu[si]), int(cu[si + 1])
        L = b - a
        qs = q[a:b].transpose(0, 1)                                  # [nh, L, hd]
        ks = k[a:b].transpose(0, 1).repeat_interleave(nh // kv, dim=0)
        vs = v[a:b].transpose(0, 1).repeat_interleave(nh // kv, dim=0)
        sc = qs @ ks.transpose(1, 2) / math.sqrt(hd)
        mask = torch.triu(torch.ones(L, L, dtype=torch.bool), diagonal=1)
        sc = sc.masked_fill(mask, float("-inf"))
        p = torch.softmax(sc, dim=-1)
        out.append((p @ vs).transpose(0, 1))                         # [L, nh, hd]
    return bf16r(torch.cat(out, dim=0))


def swiglu(g: torch.Tensor, u: torch.Tensor) -> torch.Tensor:
    """h = bf16(silu(g) * u), silu(g) = g / (1 + exp(-g))."""
    return bf16r(g / (1.0 + torch.exp(-g)) * u)


def positions(cu: Sequence[int]) -> torch.Tensor:
    return torch.cat([torch.arange(int(cu[i + 1]) - int(cu[i])) for i in range(len(cu) - 1)])


def decoder_layer(x: torch.Tensor, lw: LayerWeights, ad: Optional[Adapter], cfg, cu,
                  adapter_on: bool = True, trace: Optional[Dict] = None) -> torch.Tensor:
    """One pre-norm decoder layer; returns the layer output (bf16 values)."""
    T = x.shape[0]
    nh, kv, hd = cfg.heads, cfg.kv_heads, cfg.head_dim
    s = cfg.lora_scale
    n1 = rmsnorm(x, lw.w1, cfg.eps)
    use = adapter_on and ad is not None
    q = linear(n1, lw.wq, (lora_u(n1, ad.aq, s), ad.bq) if use else None)
    k = linear(n1, lw.wk)
    v = linear(n1, lw.wv, (lora_u(n1, ad.av, s), ad.bv) if use else None)
    pos = positions(cu)
    qr = rope(q.view(T, nh, hd), pos, cfg.rope_theta)
    kr = rope(k.view(T, kv, hd), pos, cfg.rope_theta)
    o = attention(qr, kr, v.view(T, kv, hd), cu).reshape(T, nh * hd)
    x1 = linear(o, lw.wo, residual=x)
    n2 = rmsnorm(x1, lw.w2, cfg.eps)
    g = linear(n2, lw.wg)
    u = linear(n2, lw.wu)
    h = swiglu(g, u)
    out = linear(h, lw.wd, residual=x1)
    if trace is not None:
        trace.update(n1=n1, q=q, k=k, v=v, qr=qr, kr=kr, o=o, x1=x1, n2=n2, g=g, u=u, h=h, out=out)
    return out


# --------------------------------------------------------------------------- stack

@dataclasses.dataclass
class StackWeights:
    layers: List[LayerWeights]
    embed: torch.Tensor       # [V, H] dequantised
    lm_head: torch.Tensor     # [V, H] dequantised (same tensor when tied)
    wf: torch.Tensor          # final norm weight [H]


def targets(tokens: np.ndarray, cu: Sequence[int]) -> np.ndarray:
    """Next-token target of each position (-1 at the last position of a sequence)."""
    y = np.full(len(tokens), -1, np.int64)
    for i in range(len(cu) - 1):
        a, b = int(cu[i]), int(cu[i + 1])
        y[a:b - 1] = tokens[a + 1:b]
    return y


def stack_forward(tokens: np.ndarray, cu, sw: StackWeights, adapters: Optional[List[Adapter]],
                  cfg, adapter_on: bool = True, trace: Optional[Dict] = None) -> Dict:
    """embed -> layers -> final RMSNorm -> logits -> log-sum-exp -> per-token logprobs.

    Returns lp [T] (0 where there is no target), lse [T], final hidden hf [T, H].
    """
    x = sw.embed[torch.from_numpy(tokens.astype(np.int64))]
    xs = [x]
    for li, lw in enumerate(sw.layers):
        x = decoder_layer(x, lw, adapters[li] if adapters else None, cfg, cu, adapter_on)
        xs.append(x)
    hf = rmsnorm(x, sw.wf, cfg.eps)
    logits = hf @ sw.lm_head.T
    lse = torch.logsumexp(logits, dim=-1)
    y = targets(tokens, cu)
    has = torch.from_numpy(y >= 0)
    yt = torch.from_numpy(np.where(y >= 0, y, 0))
    lp = torch.where(has, logits.gather(1, yt[:, None])[:, 0] - lse, torch.zeros((), dtype=F64))
    if trace is not None:
        trace.update(xs=xs, hf=hf, logits=logits)
    return dict(lp=lp, lse=lse, hf=hf)


def seq_sums(lp: torch.Tensor, mask: np.ndarray, cu) -> torch.Tensor:
    m = torch.from_numpy(mask.astype(np.float64))
    return torch.stack([(lp * m)[int(cu[i]):int(cu[i + 1])].sum() for i in range(len(cu) - 1)])


def sft_loss(lp: torch.Tensor, mask: np.ndarray) -> torch.Tensor:
    """Mean negative log-likelihood over the positions the mask selects."""
    m = torch.from_numpy(mask.astype(np.float64))
    return -(lp * m).sum() / m.sum()


def dpo_loss(pi: torch.Tensor, ref: torch.Tensor, beta: float) -> torch.Tensor:
    """Mean over pairs of -log sigmoid(beta ((pi_c - ref_c) - (pi_r - ref_r))).

    Sequences come as (chosen, rejected) pairs; -log sigmoid(z) = softplus(-z).
    """
    z = beta * ((pi[0::2] - ref[0::2]) - (pi[1::2] - ref[1::2]))
    return F.softplus(-z).mean()


# ---------------------------------------------------------------- other preference losses
# The pages list ORPO, SimPO and KTO beside DPO as methods run over the streamed base
# (axbrief.com, "The Architecture of Low-VRAM Alignment"; evermx.com summary) without
# defining them; these follow the methods' own papers.  All act on per-sequence
# logprob sums over the response positions, as DPO does.

def seq_counts(mask: np.ndarray, cu) -> torch.Tensor:
    """Number of response positions (mask = 1) of each sequence."""
    return torch.tensor([float(mask[int(cu[i]):int(cu[i + 1])].sum()) for i in range(len(cu) - 1)],
                        dtype=torch.float64)


def simpo_loss(pi: torch.Tensor, counts: torch.Tensor, beta: float, gamma: float) -> torch.Tensor:
    """SimPO (Meng, Xia, Chen 2024): mean over pairs of
    -log sigmoid(beta pi_c / |c| - beta pi_r / |r| - gamma); no reference model."""
    avg = pi / counts.to(pi.dtype)
    z = beta * (avg[0::2] - avg[1::2]) - gamma
    return F.softplus(-z).mean()


def orpo_loss(pi: torch.Tensor, counts: torch.Tensor, lam: float) -> torch.Tensor:
    """ORPO (Hong, Lee, Thorne 2024): mean over pairs of the chosen response's mean NLL
    plus lam * -log sigmoid(log odds(c) - log odds(r)), where odds(y) = P / (1 - P) and
    P = exp(mean logprob of y); no reference model."""
    avg = pi / counts.to(pi.dtype)
    log_odds = avg - torch.log1p(-torch.exp(avg))
    nll = -avg[0::2]
    return (nll + lam * F.softplus(-(log_odds[0::2] - log_odds[1::2]))).mean()


def kto_loss(pi: torch.Tensor, ref: torch.Tensor, desirable: torch.Tensor, beta: float, lam_d: float,
             lam_u: float) -> torch.Tensor:
    """KTO (Ethayarajh et al. 2024): r = pi - ref per sequence, reference point
    z0 = max(0, mean r over the batch) taken without gradient; loss = mean of
    lam_d (1 - sigmoid(beta (r - z0))) on desirable sequences and
    lam_u (1 - sigmoid(beta (z0 - r))) on undesirable ones."""
    r = pi - ref
    z0 = torch.clamp(r.detach().mean(), min=0.0)
    d = desirable.to(torch.bool)
    v = torch.where(d, lam_d * torch.sigmoid(beta * (r - z0)), lam_u * torch.sigmoid(beta * (z0 - r)))
    lam = torch.where(d, torch.full_like(r, lam_d), torch.full_like(r, lam_u))
    return (lam - v).mean()


def pair_desirable(nseq: int) -> torch.Tensor:
    """KTO labels for (chosen, rejected) pair data: chosen desirable, rejected not."""
    return torch.tensor([1 - (i % 2) for i in range(nseq)], dtype=torch.uint8)


def train_step(tokens: np.ndarray, cu, mask: np.ndarray, sw: StackWeights,
               adapters: List[Adapter], cfg, method: Optional[str] = None) -> Dict:
    """One SFT, DPO, SimPO, ORPO or KTO step: loss, logprobs and the LoRA gradients (fp64).

    The base is frozen; gradients are taken for A and B of every layer only.
    """
    method = method or cfg.method
    for ad in adapters:
        for p in ad.params():
            p.requires_grad_(True)
            p.grad = None
    pol = stack_forward(tokens, cu, sw, adapters, cfg, adapter_on=True)
    out = dict(lp=pol["lp"].detach(), lse=pol["lse"].detach())
    if method == "sft":
        loss = sft_loss(pol["lp"], mask)
    elif method in ("simpo", "orpo"):
        pi = seq_sums(pol["lp"], mask, cu)
        counts = seq_counts(mask, cu)
        if method == "simpo":
            loss = simpo_loss(pi, counts, cfg.beta, getattr(cfg, "simpo_gamma", 1.0))
        else:
            loss = orpo_loss(pi, counts, getattr(cfg, "orpo_lambda", 0.1))
        out.update(pi=pi.detach())
    else:
        with torch.no_grad():
            ref = stack_forward(tokens, cu, sw, adapters, cfg, adapter_on=False)
        pi = seq_sums(pol["lp"], mask, cu)
        rs = seq_sums(ref["lp"], mask, cu)
        if method == "kto":
            loss = kto_loss(pi, rs, pair_desirable(len(cu) - 1), cfg.beta, getattr(cfg, "kto_lambda_d", 1.0),
                            getattr(cfg, "kto_lambda_u", 1.0))
        else:
            loss = dpo_loss(pi, rs, cfg.beta)
        out.update(lp_ref=ref["lp"], pi=pi.detach(), ref=rs)
    loss.backward()
    out["loss"] = loss.detach()
    out["grads"] = [[p.grad.clone() for p in ad.params()] for ad in adapters]
    return out


# --------------------------------------------------------------------------- building inputs

def build_stack(cfg, seed: int = 0, synth=None) -> StackWeights:
    """Dequantised base of a stack config from the shared seeded draws."""
    layers = []
    for l in range(cfg.layers):
        w = {n: dequant_weight(synth.weight(cfg, l, n, seed))
             for n in ("q", "k", "v", "o", "gate", "up", "down")}
        layers.append(LayerWeights(w["q"], w["k"], w["v"], w["o"], w["gate"], w["up"], w["down"],
                                   t64(synth.norm_weight(cfg, l, 0, seed)),
                                   t64(synth.norm_weight(cfg, l, 1, seed))))
    emb = dequant_weight(synth.weight(cfg, -1, "embed", seed))
    head = emb if cfg.tied else dequant_weight(synth.weight(cfg, -1, "lm_head", seed))
    return StackWeights(layers, emb, head, t64(synth.norm_weight(cfg, -1, 0, seed)))


def cast_stack(sw: StackWeights, dtype) -> StackWeights:
    """The same dequantised base in another floating type (see accumulate_in)."""
    layers = [LayerWeights(*[getattr(l, f.name).to(dtype) for f in dataclasses.fields(LayerWeights)])
              for l in sw.layers]
    head = sw.lm_head.to(dtype)
    emb = head if sw.embed is sw.lm_head else sw.embed.to(dtype)
    return StackWeights(layers, emb, head, sw.wf.to(dtype))


def cast_adapters(ads: List[Adapter], dtype) -> List[Adapter]:
    return [Adapter(*[p.detach().to(dtype) for p in a.params()]) for a in ads]


def build_adapters(cfg, seed: int = 0, synth=None, zero_b: bool = False) -> List[Adapter]:
    ads = []
    for l in range(cfg.layers):
        aq, bq = synth.lora_weights(cfg, l, "q", seed, zero_b=zero_b)
        av, bv = synth.lora_weights(cfg, l, "v", seed, zero_b=zero_b)
        ads.append(Adapter(t64(aq), t64(bq), t64(av), t64(bv)))
    return ads


# --------------------------------------------------------------------------- single linear

def lora_linear_step(x: np.ndarray, w_deq: np.ndarray, a: np.ndarray, b: np.ndarray, s: float,
                     dy: np.ndarray) -> Dict:
    """Single NF4 LoRA linear, forward and backward for the loss sum(Y * dY).

    Y = bf16(X W^T + u B^T), u = bf16(s X A^T); returns Y, dX, dA, dB (fp64).
    """
    X = t64(x).requires_grad_(True)
    A = t64(a).requires_grad_(True)
    B = t64(b).requires_grad_(True)
    y = linear(X, t64(w_deq), (lora_u(X, A, s), B))
    (y * t64(dy)).sum().backward()
    return dict(y=y.detach(), dx=X.grad, da=A.grad, db=B.grad)


# --------------------------------------------------------------------------- optimizer

def adamw_update(p: torch.Tensor, g: torch.Tensor, m: torch.Tensor, v: torch.Tensor, step: int, lr: float,
                 beta1: float, beta2: float, eps: float, weight_decay: float) -> None:
    """One AdamW step in place (fp64): decoupled weight decay p -= lr wd p, then the
    bias-corrected Adam update (Loshchilov & Hutter 2019).  The pages only say the
    optimizer is picked automatically; this is the usual choice for LoRA."""
    p.mul_(1.0 - lr * weight_decay)
    m.mul_(beta1).add_((1.0 - beta1) * g)
    v.mul_(beta2).add_((1.0 - beta2) * g * g)
    mh = m / (1.0 - beta1 ** step)
    vh = v / (1.0 - beta2 ** step)
    p.sub_(lr * mh / (torch.sqrt(vh) + eps))
