"""Seeded synthetic inputs shared by the CUDA path, the oracle and the benchmark.

This module holds only shapes and random draws: no NF4 quantisation, no model
arithmetic.  Every array is a pure function of (config, seed, tensor id), so a
single matrix of a 32-layer stack can be regenerated on its own.

Shapes follow the five workloads of the layer-streamed LoRA fine-tuning method
described on the Soup pages ("The Core Idea: Layer Streaming" on lucaberton.com;
the evermx.com summary): a single NF4 LoRA linear, one Llama-style decoder layer,
and Qwen2.5-3B / Llama-3.1-8B / Qwen2.5-32B shaped stacks.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Tuple

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class StackConfig:
    """Shape of a Llama-style decoder stack (no biases, pre-norm, SwiGLU)."""
    name: str
    layers: int
    hidden: int
    heads: int
    kv_heads: int
    head_dim: int
    inter: int
    vocab: int
    tied: bool
    rope_theta: float
    eps: float
    lora_r: int = 16
    lora_alpha: float = 32.0
    seq_len: int = 512            # tokens per sequence
    nseq: int = 1                 # sequences per pass
    prompt_len: int = 0           # DPO: shared prompt length (0 = SFT)
    method: str = "sft"           # "sft" | "dpo" | "simpo" | "orpo" | "kto"
    beta: float = 0.1
    simpo_gamma: float = 1.0      # SimPO target margin
    orpo_lambda: float = 0.1      # ORPO odds-ratio weight
    kto_lambda_d: float = 1.0     # KTO weights of desirable / undesirable sequences
    kto_lambda_u: float = 1.0
    cap_bytes: int = 0            # device cap (0 = none)

    @property
    def tokens(self) -> int:
        return self.seq_len * self.nseq

    @property
    def n_q(self) -> int:
        return self.heads * self.head_dim

    @property
    def n_kv(self) -> int:
        return self.kv_heads * self.head_dim

    @property
    def lora_scale(self) -> float:
        return self.lora_alpha / self.lora_r

    def with_(self, **kw) -> "StackConfig":
        return dataclasses.replace(self, **kw)


# Single NF4 LoRA linear, fwd+bwd (d_in = d_out = 256, 64 tokens, r = 8, alpha = 16).
LINEAR_256 = dict(d_in=256, d_out=256, tokens=64, r=8, alpha=16.0)

# One Llama-style decoder layer at the Qwen2.5-0.5B width, SFT over 512 tokens.
# Its loss wraps the layer in the 0.5B tied vocabulary.
LAYER_896 = StackConfig("layer-896", layers=1, hidden=896, heads=14, kv_heads=2, head_dim=64,
                        inter=4864, vocab=151936, tied=True, rope_theta=1e6, eps=1e-6,
                        seq_len=512, nseq=1)

# Qwen2.5-3B-shaped stack, SFT, batch 1 x 512.
QWEN_3B = StackConfig("qwen2.5-3b", layers=36, hidden=2048, heads=16, kv_heads=2, head_dim=128,
                      inter=11008, vocab=151936, tied=True, rope_theta=1e6, eps=1e-6,
                      seq_len=512, nseq=1)

# Llama-3.1-8B-shaped stack, DPO (beta 0.1): one pair, 256-token shared prompt and
# 256-token responses, so one pass carries 2 x 512 tokens.
LLAMA_8B = StackConfig("llama-3.1-8b", layers=32, hidden=4096, heads=32, kv_heads=8, head_dim=128,
                       inter=14336, vocab=128256, tied=False, rope_theta=5e5, eps=1e-5,
                       seq_len=512, nseq=2, prompt_len=256, method="dpo", beta=0.1)

# Qwen2.5-32B-shaped stack, DPO (beta 0.1), 2 x 1024 tokens (512 prompt + 512
# response per sequence) under a 4 GiB device cap.
QWEN_32B = StackConfig("qwen2.5-32b", layers=64, hidden=5120, heads=40, kv_heads=8, head_dim=128,
                       inter=27648, vocab=152064, tied=False, rope_theta=1e6, eps=1e-6,
                       seq_len=1024, nseq=2, prompt_len=512, method="dpo", beta=0.1,
                       cap_bytes=4 << 30)

CONFIGS: Dict[str, StackConfig] = {c.name: c for c in (LAYER_896, QWEN_3B, LLAMA_8B, QWEN_32B)}

# Frozen matrices of one decoder layer, in the order the device slot holds them.
# q, k, v are stacked into one [n_q + 2 n_kv, H] matrix; gate and up into [2I, H].
MATRIX_IDS = {"q": 0, "k": 1, "v": 2, "o": 3, "gate": 4, "up": 5, "down": 6,
              "embed": 7, "lm_head": 8}


def matrix_shape(cfg: StackConfig, name: str) -> Tuple[int, int]:
    H, I = cfg.hidden, cfg.inter
    return {"q": (cfg.n_q, H), "k": (cfg.n_kv, H), "v": (cfg.n_kv, H), "o": (H, cfg.n_q),
            "gate": (I, H), "up": (I, H), "down": (H, I),
            "embed": (cfg.vocab, H), "lm_head": (cfg.vocab, H)}[name]


def _rng(seed: int, *ids: int) -> np.random.Generator:
    return np.random.default_rng([seed, *ids])


def to_bf16_values(x: np.ndarray) -> np.ndarray:
    """Store an fp32 draw as bf16 (the inputs' dtype); returns fp32 holding bf16 values."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


ROW_BLOCK = 256


def weight(cfg: StackConfig, layer: int, name: str, seed: int = 0, row0: int = 0,
           nrows: int = -1, std: float = 0.02) -> np.ndarray:
    """Frozen fp32 weight W ~ N(0, std), rows [row0, row0 + nrows) of the [N, K] matrix.

    Drawn in independent 256-row blocks (one generator per block) so any rows of a
    large matrix can be regenerated without the rest.  layer = -1 for embed/lm_head.
    """
    n, k = matrix_shape(cfg, name)
    end = n if nrows < 0 else row0 + nrows
    out = np.empty((end - row0, k), np.float32)
    for blk in range(row0 // ROW_BLOCK, (end + ROW_BLOCK - 1) // ROW_BLOCK):
        r0 = blk * ROW_BLOCK
        g = _rng(seed, 1, layer + 1, MATRIX_IDS[name], blk)
        b = g.standard_normal((min(ROW_BLOCK, n - r0), k), dtype=np.float32)
        lo, hi = max(r0, row0), min(r0 + b.shape[0], end)
        out[lo - row0: hi - row0] = b[lo - r0: hi - r0]
    out *= np.float32(std)
    return out


def norm_weight(cfg: StackConfig, layer: int, which: int, seed: int = 0) -> np.ndarray:
    """RMSNorm weight 1 + 0.1 N(0,1) as bf16 values; which 0/1 = attn/mlp, layer -1 = final."""
    g = _rng(seed, 3, layer + 1, which)
    return to_bf16_values(1.0 + 0.1 * g.standard_normal(cfg.hidden, dtype=np.float32))


def lora_weights(cfg: StackConfig, layer: int, proj: str, seed: int = 0,
                 std: float = 0.01, zero_b: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """LoRA A [r, K] and B [N, r] ~ N(0, std) as bf16 values (proj in {"q", "v"})."""
    n, k = matrix_shape(cfg, proj)
    g = _rng(seed, 4, layer + 1, MATRIX_IDS[proj])
    a = to_bf16_values(std * g.standard_normal((cfg.lora_r, k), dtype=np.float32))
    b = to_bf16_values(std * g.standard_normal((n, cfg.lora_r), dtype=np.float32))
    if zero_b:
        b = np.zeros_like(b)
    return a, b


def tokens(cfg: StackConfig, seed: int = 0) -> np.ndarray:
    """Token ids for one pass, int32 [T]; uniform over the vocabulary.

    Preference methods: sequences come in (chosen, rejected) pairs that share their
    first prompt_len tokens.
    """
    g = _rng(seed, 5)
    t = g.integers(0, cfg.vocab, size=(cfg.nseq, cfg.seq_len), dtype=np.int64)
    if cfg.method != "sft" and cfg.prompt_len > 0:
        for p in range(0, cfg.nseq, 2):
            t[p + 1, :cfg.prompt_len] = t[p, :cfg.prompt_len]
    return t.reshape(-1).astype(np.int32)


def seq_offsets(cfg: StackConfig) -> np.ndarray:
    """Cumulative sequence starts, int32 [nseq + 1]."""
    return (np.arange(cfg.nseq + 1) * cfg.seq_len).astype(np.int32)


def loss_mask(cfg: StackConfig) -> np.ndarray:
    """uint8 [T]: 1 where position t's prediction of token t+1 counts.

    SFT: every position but the last of each sequence.  Preference methods: only
    predictions of response tokens (positions prompt_len-1 .. seq_len-2 of each sequence).
    """
    m = np.zeros((cfg.nseq, cfg.seq_len), np.uint8)
    lo = cfg.prompt_len - 1 if cfg.method != "sft" and cfg.prompt_len > 0 else 0
    m[:, lo: cfg.seq_len - 1] = 1
    return m.reshape(-1)


def gaussian(shape, seed: int, *ids: int, std: float = 1.0) -> np.ndarray:
    """N(0, std) fp32 draw, stored as bf16 values."""
    g = _rng(seed, 6, *ids)
    return to_bf16_values(std * g.standard_normal(shape, dtype=np.float32))


def gaussian_f32(shape, seed: int, *ids: int, std: float = 1.0) -> np.ndarray:
    g = _rng(seed, 7, *ids)
    return (std * g.standard_normal(shape, dtype=np.float32)).astype(np.float32)


def small_stack(base: StackConfig, layers: int, vocab: int, seq_len: int, nseq: int = 1,
                prompt_len: int = 0, **kw) -> StackConfig:
    """A reduced copy of a stack shape for parity runs the oracle finishes quickly."""
    return base.with_(name=f"{base.name}-L{layers}-V{vocab}-S{seq_len}x{nseq}", layers=layers,
                      vocab=vocab, seq_len=seq_len, nseq=nseq, prompt_len=prompt_len, **kw)
