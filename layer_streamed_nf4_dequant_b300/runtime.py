"""Host-side plumbing around libls: pinned layer images, workspace, adapters, steps.

PyTorch supplies device memory, pinned host memory and streams; every step of the
computation runs inside libls.so.  The frozen base is held in pinned host RAM in
the library's slot layout (one buffer per layer, so each layer read is one
host-to-device copy), as the layer-streaming design on the Soup pages prescribes
("The Core Idea: Layer Streaming", Soup: Fine-Tune an 8B Model on a 4 GB GPU).
"""
from __future__ import annotations

import contextlib
import ctypes as C
import functools
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, List, Optional

import numpy as np
import torch

from ._binding import (LSError, call, check, last_error, lib, ls_config, ls_layer_host, ls_nf4_host, ls_stats_t,
                       ls_vocab_host, lsk_gemm_plan)

MATS = ("q", "k", "v", "o", "gate", "up", "down")


def _stream_ordered(fn):
    """Run a Stack method's library calls in stream order with the caller (Stack._ordered)."""
    @functools.wraps(fn)
    def wrapper(self, *args, **kwargs):
        with self._ordered():
            return fn(self, *args, **kwargs)
    return wrapper


def gemm_plan(mode: int, M: int, N: int, K: int, ext_k: int = 0, split: int = 0, pair_rows: int = 0,
              with_workspace: bool = True, force_bn: int = 0, force_nacc: int = 0, sms: int = 148) -> Dict:
    """Tile shape and schedule the library picks for one NF4 product (lsk_nf4_gemm_plan;
    host only).  mode 0: out [M, N] = A [M, K] . deq(W)^T; mode 1: out [M, K] = A [M, N] . deq(W)."""
    p = lsk_gemm_plan()
    check(lib().lsk_nf4_gemm_plan(mode, M, N, K, ext_k, split, pair_rows, int(with_workspace), force_bn, force_nacc,
                                  sms, C.byref(p)))
    return p.as_dict()


def make_config(s, max_tokens: int = 0, max_seqs: int = 0, max_seq_len: int = 0, resident: bool = False,
                cap_bytes: Optional[int] = None, vocab_chunk_rows: int = 0, dpo_shared_read: bool = False) -> ls_config:
    """ls_config from a stack shape (anything with the synth.StackConfig fields)."""
    c = ls_config()
    c.layers, c.hidden, c.heads, c.kv_heads, c.head_dim = s.layers, s.hidden, s.heads, s.kv_heads, s.head_dim
    c.inter, c.vocab, c.tied, c.lora_r = s.inter, s.vocab, int(s.tied), s.lora_r
    c.lora_scale, c.rope_theta, c.eps = s.lora_alpha / s.lora_r, s.rope_theta, s.eps
    c.max_tokens = max_tokens or s.seq_len * s.nseq
    c.max_seqs = max_seqs or s.nseq
    c.max_seq_len = max_seq_len or s.seq_len
    c.vocab_chunk_rows = vocab_chunk_rows
    c.resident = int(resident)
    c.dpo_shared_read = int(dpo_shared_read)
    c.cap_bytes = s.cap_bytes if cap_bytes is None else cap_bytes
    return c


def plan_bytes(cfg: ls_config) -> int:
    n = C.c_uint64(0)
    check(lib().ls_plan(C.byref(cfg), C.byref(n)))
    return n.value


def layer_layout(cfg: ls_config):
    offs = (C.c_uint64 * 16)()
    nb = C.c_uint64(0)
    check(lib().ls_layer_layout(C.byref(cfg), offs, C.byref(nb)))
    return [int(o) for o in offs], nb.value


def quantize_host(w: np.ndarray, packed: Optional[np.ndarray] = None, absmax: Optional[np.ndarray] = None,
                  nthreads: int = 0):
    """NF4-quantise fp32 W [N, K] with the library's host quantiser."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    if packed is None:
        packed = np.empty((n, k // 2), np.uint8)
    if absmax is None:
        absmax = np.empty((n, k // 64), np.float32)
    check(lib().nf4_quantize(w.ctypes.data, n, k, packed.ctypes.data, absmax.ctypes.data, nthreads))
    return packed, absmax


def _pinned(nbytes: int) -> torch.Tensor:
    return torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)


class Stack:
    """A libls context for one stack shape, with its pinned base, adapters and buffers."""

    def __init__(self, s, max_tokens: int = 0, max_seqs: int = 0, max_seq_len: int = 0, resident: bool = False,
                 cap_bytes: Optional[int] = None, vocab_chunk_rows: int = 0, device: str = "cuda:0",
                 dpo_shared_read: Optional[bool] = None):
        """dpo_shared_read: run the policy and reference forward of DPO / KTO in one
        sweep of the streamed layers (None: whenever the workload needs a reference
        pass and the larger forward workspace fits the device cap)."""
        self.s = s
        self.dev = torch.device(device)
        if dpo_shared_read is None:
            dpo_shared_read = False
            if getattr(s, "method", "sft") in ("dpo", "kto"):
                trial = make_config(s, max_tokens, max_seqs, max_seq_len, resident, cap_bytes, vocab_chunk_rows, True)
                n = C.c_uint64(0)
                dpo_shared_read = lib().ls_plan(C.byref(trial), C.byref(n)) == 0
        self.shared_read = bool(dpo_shared_read)
        self.cfg = make_config(s, max_tokens, max_seqs, max_seq_len, resident, cap_bytes, vocab_chunk_rows,
                               self.shared_read)
        self.ws_bytes = plan_bytes(self.cfg)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.dev)
        self.compute = torch.cuda.Stream(self.dev)
        self.copy = torch.cuda.Stream(self.dev)
        h = C.c_void_p()
        check(lib().ls_create(C.byref(self.cfg), self.ws.data_ptr(), self.ws_bytes, self.compute.cuda_stream,
                              self.copy.cuda_stream, C.byref(h)))
        self.ctx = h.value
        self.offs, self.img_bytes = layer_layout(self.cfg)
        self.images: List[torch.Tensor] = []
        self.vocab_bufs: Dict[str, torch.Tensor] = {}
        self.adapters: List[Dict[str, torch.Tensor]] = []
        self._keep = []

    # ------------------------------------------------------------------ loading
    @contextlib.contextmanager
    def _ordered(self):
        """The library runs on the stack's own compute stream while callers make and free
        tensors on their current stream.  Join the two around every call that queues device
        work: the compute stream first waits for what the caller queued (uploads of the
        tokens, offsets and mask, adapter factors), and the caller's stream then waits for
        the stack's work, so its outputs are ready there and the caching allocator cannot
        hand a tensor the library still reads or writes to a new owner."""
        cur = torch.cuda.current_stream(self.dev)
        if cur == self.compute:
            yield
            return
        self.compute.wait_stream(cur)
        try:
            yield
        finally:
            cur.wait_stream(self.compute)

    def _shape(self, name):
        s = self.s
        H, I, nq, nkv = s.hidden, s.inter, s.heads * s.head_dim, s.kv_heads * s.head_dim
        return {"q": (nq, H), "k": (nkv, H), "v": (nkv, H), "o": (H, nq), "gate": (I, H), "up": (I, H),
                "down": (H, I)}[name]

    def load_layer_arrays(self, layer: int, weights: Dict[str, np.ndarray], attn_norm: np.ndarray,
                          mlp_norm: np.ndarray, nthreads: int = 0):
        """Quantise fp32 weights into a pinned image in slot layout and register it."""
        img = _pinned(self.img_bytes)
        buf = img.numpy()
        for m, name in enumerate(MATS):
            n, k = self._shape(name)
            pk = buf[self.offs[m]: self.offs[m] + n * k // 2].reshape(n, k // 2)
            am = buf[self.offs[7 + m]: self.offs[7 + m] + n * (k // 64) * 4].view(np.float32).reshape(n, k // 64)
            quantize_host(weights[name], pk, am, nthreads)
        H = self.s.hidden
        buf[self.offs[14]: self.offs[14] + 2 * H] = _bf16_bytes(attn_norm)
        buf[self.offs[15]: self.offs[15] + 2 * H] = _bf16_bytes(mlp_norm)
        self._register_layer(layer, img)

    def _register_layer(self, layer: int, img: torch.Tensor):
        base = img.data_ptr()
        lh = ls_layer_host()
        for m, name in enumerate(MATS):
            setattr(lh, name, ls_nf4_host(base + self.offs[m], base + self.offs[7 + m]))
        lh.attn_norm = base + self.offs[14]
        lh.mlp_norm = base + self.offs[15]
        check(lib().load_layer_nf4(self.ctx, layer, C.byref(lh)), self.ctx)
        while len(self.images) <= layer:
            self.images.append(None)
        self.images[layer] = img

    def load_vocab_arrays(self, embed: np.ndarray, lm_head: Optional[np.ndarray], final_norm: np.ndarray,
                          nthreads: int = 0):
        V, H = embed.shape
        ep = _pinned(V * H // 2)
        ea = _pinned(V * (H // 64) * 4)
        quantize_host(embed, ep.numpy().reshape(V, H // 2), ea.numpy().view(np.float32).reshape(V, H // 64), nthreads)
        self.vocab_bufs = {"ep": ep, "ea": ea}
        vh = ls_vocab_host()
        vh.embed = ls_nf4_host(ep.data_ptr(), ea.data_ptr())
        if not self.s.tied:
            hp = _pinned(V * H // 2)
            ha = _pinned(V * (H // 64) * 4)
            quantize_host(lm_head, hp.numpy().reshape(V, H // 2), ha.numpy().view(np.float32).reshape(V, H // 64),
                          nthreads)
            self.vocab_bufs.update(hp=hp, ha=ha)
            vh.lm_head = ls_nf4_host(hp.data_ptr(), ha.data_ptr())
        fn = _pinned(2 * H)
        fn.numpy()[:] = _bf16_bytes(final_norm)
        self.vocab_bufs["fn"] = fn
        vh.final_norm = fn.data_ptr()
        check(lib().load_vocab_nf4(self.ctx, C.byref(vh)), self.ctx)

    def load_synthetic(self, synth, seed: int = 0, workers: int = 0):
        """Draw the base from the shared seeded generators and load it (threads over layers)."""
        s = self.s
        workers = workers or min(16, os.cpu_count() or 1)

        def one(layer):
            w = {n: synth.weight(s, layer, n, seed) for n in MATS}
            self.load_layer_arrays(layer, w, synth.norm_weight(s, layer, 0, seed),
                                   synth.norm_weight(s, layer, 1, seed), nthreads=1)

        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(one, range(s.layers)))
        emb = synth.weight(s, -1, "embed", seed)
        head = None if s.tied else synth.weight(s, -1, "lm_head", seed)
        self.load_vocab_arrays(emb, head, synth.norm_weight(s, -1, 0, seed))

    def adopt_base(self, other: "Stack"):
        """Register another Stack's pinned host base (same shape) instead of loading a copy."""
        if other.img_bytes != self.img_bytes or other.s.layers != self.s.layers:
            raise ValueError("adopt_base: stack shapes differ")
        for layer, img in enumerate(other.images):
            self._register_layer(layer, img)
        vb = other.vocab_bufs
        vh = ls_vocab_host()
        vh.embed = ls_nf4_host(vb["ep"].data_ptr(), vb["ea"].data_ptr())
        if not self.s.tied:
            vh.lm_head = ls_nf4_host(vb["hp"].data_ptr(), vb["ha"].data_ptr())
        vh.final_norm = vb["fn"].data_ptr()
        check(lib().load_vocab_nf4(self.ctx, C.byref(vh)), self.ctx)
        self.vocab_bufs = dict(vb)

    # ------------------------------------------------------------------ file-backed layers
    def layer_file_stride(self) -> int:
        """Bytes between consecutive layer images in a layer file (4 KiB-aligned)."""
        return (self.img_bytes + 4095) // 4096 * 4096

    def write_layer_file(self, path: str):
        """Write every pinned layer image to one file (layer l at l * layer_file_stride())."""
        stride = self.layer_file_stride()
        with open(path, "wb") as f:
            for l, img in enumerate(self.images):
                f.seek(l * stride)
                f.write(img.numpy().tobytes())
            f.truncate(len(self.images) * stride)

    def use_layer_file(self, path: str, nbuf: int = 3, release_ram: bool = True):
        """Stream every decoder layer from `path` (written by write_layer_file) through
        `nbuf` pinned staging buffers instead of from pinned RAM images."""
        stride = self.layer_file_stride()
        self.staging = torch.empty(nbuf * stride, dtype=torch.uint8, pin_memory=True)
        check(lib().ls_set_staging(self.ctx, self.staging.data_ptr(), stride, nbuf), self.ctx)
        for l in range(self.s.layers):
            check(lib().load_layer_file(self.ctx, l, path.encode(), l * stride), self.ctx)
        if release_ram:
            self.images = [None] * self.s.layers

    # ------------------------------------------------------------------ adapters
    @_stream_ordered
    def set_adapter(self, layer: int, aq, bq, av, bv):
        """Bind bf16 device LoRA factors (A [r,H], B [N,r]); fp32 grads are allocated here."""
        d = {"aq": aq, "bq": bq, "av": av, "bv": bv}
        for k in list(d):
            d["g" + k] = torch.zeros(d[k].shape, dtype=torch.float32, device=self.dev)
        check(lib().ls_set_adapter(self.ctx, layer, aq.data_ptr(), bq.data_ptr(), av.data_ptr(), bv.data_ptr(),
                                   d["gaq"].data_ptr(), d["gbq"].data_ptr(), d["gav"].data_ptr(),
                                   d["gbv"].data_ptr()), self.ctx)
        while len(self.adapters) <= layer:
            self.adapters.append(None)
        self.adapters[layer] = d

    def set_adapters_synthetic(self, synth, seed: int = 0, zero_b: bool = False):
        for l in range(self.s.layers):
            aq, bq = synth.lora_weights(self.s, l, "q", seed, zero_b=zero_b)
            av, bv = synth.lora_weights(self.s, l, "v", seed, zero_b=zero_b)
            t = [torch.from_numpy(x).to(torch.bfloat16).to(self.dev) for x in (aq, bq, av, bv)]
            self.set_adapter(l, *t)

    @_stream_ordered
    def export_adapter(self, path: str):
        """Write the bound LoRA factors with canonical keys (see adapters.py)."""
        from .adapters import save_adapter
        ads = [{k: self.adapters[l][k].detach().view(torch.int16).cpu().numpy().view(np.uint16)
                for k in ("aq", "bq", "av", "bv")} for l in range(self.s.layers)]
        return save_adapter(path, ads, self.s.lora_r, self.s.lora_alpha)

    def import_adapter(self, path: str):
        """Bind the LoRA factors of a canonical-key adapter file (refuses mismatched keys)."""
        from .adapters import load_adapter
        s = self.s
        ads = load_adapter(path, s.layers, s.hidden, s.heads * s.head_dim, s.kv_heads * s.head_dim, s.lora_r)
        for l, ad in enumerate(ads):
            t = [torch.from_numpy(ad[k].view(np.int16)).view(torch.bfloat16).to(self.dev)
                 for k in ("aq", "bq", "av", "bv")]
            self.set_adapter(l, *t)

    @_stream_ordered
    def init_optimizer(self, lr: float = 1e-4, betas=(0.9, 0.999), eps: float = 1e-8, weight_decay: float = 0.0):
        """AdamW state for the bound adapters: fp32 master (from the bf16 factors) and moments."""
        n = self.grad_numel()
        self.opt = {"master": torch.empty(n, dtype=torch.float32, device=self.dev),
                    "m": torch.zeros(n, dtype=torch.float32, device=self.dev),
                    "v": torch.zeros(n, dtype=torch.float32, device=self.dev),
                    "step": 0, "lr": lr, "betas": betas, "eps": eps, "wd": weight_decay}
        check(lib().lora_params(self.ctx, self.opt["master"].data_ptr()), self.ctx)

    @_stream_ordered
    def optimizer_step(self, zero_grads: bool = True):
        """One AdamW step on every bound adapter from its accumulated gradient."""
        o = self.opt
        o["step"] += 1
        check(lib().lora_adamw(self.ctx, o["master"].data_ptr(), o["m"].data_ptr(), o["v"].data_ptr(), o["step"],
                               o["lr"], o["betas"][0], o["betas"][1], o["eps"], o["wd"], int(zero_grads)), self.ctx)

    def grad_numel(self) -> int:
        s = self.s
        return s.layers * (2 * s.lora_r * s.hidden + s.lora_r * (s.heads + s.kv_heads) * s.head_dim)

    # ------------------------------------------------------------------ steps
    def upload_batch(self, tokens: np.ndarray, cu: np.ndarray, mask: np.ndarray):
        """Device copies of one batch's token ids, sequence offsets and loss mask."""
        t = torch.from_numpy(np.ascontiguousarray(tokens, np.int32)).to(self.dev)
        c = torch.from_numpy(np.ascontiguousarray(cu, np.int32)).to(self.dev)
        m = torch.from_numpy(np.ascontiguousarray(mask, np.uint8)).to(self.dev)
        return t, c, m

    @_stream_ordered
    def fwd(self, tok, cu, mask, adapter_on: bool = True, save: bool = True, sums: Optional[torch.Tensor] = None):
        nseq = cu.numel() - 1
        self._last_rows = tok.numel()
        if sums is None:
            sums = torch.empty(nseq, dtype=torch.float32, device=self.dev)
        check(lib().stream_step_fwd(self.ctx, tok.data_ptr(), tok.numel(), nseq, cu.data_ptr(), mask.data_ptr(),
                                    int(adapter_on), int(save), sums.data_ptr()), self.ctx)
        return sums

    @_stream_ordered
    def logprobs(self, T: int = 0):
        """Per-token logprobs and log-sum-exp of the last forward (2T rows after a
        shared-read DPO forward: policy, then reference)."""
        T = getattr(self, "_last_rows", T) or T
        lp = torch.empty(T, dtype=torch.float32, device=self.dev)
        lse = torch.empty(T, dtype=torch.float32, device=self.dev)
        check(lib().seq_logprobs(self.ctx, lp.data_ptr(), lse.data_ptr()), self.ctx)
        return lp, lse

    @_stream_ordered
    def activation(self, layer: int, T: int) -> torch.Tensor:
        """Entry `layer` (0..L) of the activation store of the last saved forward, bf16 [T, H]."""
        out = torch.empty((T, self.s.hidden), dtype=torch.bfloat16, device=self.dev)
        check(lib().ls_read_activation(self.ctx, layer, out.data_ptr()), self.ctx)
        return out

    def capture_reference(self, on: bool = True) -> Optional[torch.Tensor]:
        """Keep the reference rows of every activation-store entry of later shared-read
        forwards in a device buffer [(L+1), max_tokens, H] bf16 (ls_capture_reference);
        entry l of a T-token step is buffer.view(-1)[l*T*H:(l+1)*T*H].  on=False stops."""
        if not on:
            check(lib().ls_capture_reference(self.ctx, None, 0), self.ctx)
            self.ref_capture = None
            return None
        n = (self.s.layers + 1) * self.cfg.max_tokens * self.s.hidden
        self.ref_capture = torch.empty(n, dtype=torch.bfloat16, device=self.dev)
        check(lib().ls_capture_reference(self.ctx, self.ref_capture.data_ptr(), 2 * n), self.ctx)
        return self.ref_capture

    @_stream_ordered
    def bwd(self, coeffs: torch.Tensor):
        check(lib().stream_step_bwd(self.ctx, coeffs.data_ptr()), self.ctx)

    @_stream_ordered
    def fwd_dpo(self, tok, cu, mask, pi: torch.Tensor, ref: torch.Tensor):
        """Policy and reference forward in one sweep (needs a shared-read context)."""
        check(lib().stream_step_fwd_dpo(self.ctx, tok.data_ptr(), tok.numel(), cu.numel() - 1, cu.data_ptr(),
                                        mask.data_ptr(), pi.data_ptr(), ref.data_ptr()), self.ctx)
        self._last_rows = 2 * tok.numel()

    @_stream_ordered
    def dpo_step(self, tok, cu, mask, beta: float, out: Optional[Dict] = None) -> Dict:
        """Policy pass (adapter on, store kept) and reference pass (adapter off) -- one
        shared sweep of the layers, or two -- then the DPO loss and the backward."""
        nseq = cu.numel() - 1
        o = out if out is not None else {
            "pi": torch.empty(nseq, dtype=torch.float32, device=self.dev),
            "ref": torch.empty(nseq, dtype=torch.float32, device=self.dev),
            "loss": torch.empty(1, dtype=torch.float32, device=self.dev),
            "coeffs": torch.empty(nseq, dtype=torch.float32, device=self.dev)}
        if self.shared_read:
            self.fwd_dpo(tok, cu, mask, o["pi"], o["ref"])
        else:
            self.fwd(tok, cu, mask, True, True, o["pi"])
            self.fwd(tok, cu, mask, False, False, o["ref"])
        check(lib().dpo_loss(self.ctx, o["pi"].data_ptr(), o["ref"].data_ptr(), nseq // 2, beta,
                             o["loss"].data_ptr(), o["coeffs"].data_ptr()), self.ctx)
        self.bwd(o["coeffs"])
        return o

    @_stream_ordered
    def pref_step(self, method: str, tok, cu, mask, out: Optional[Dict] = None) -> Dict:
        """One preference-optimisation step on (chosen, rejected) pairs: "dpo", "kto"
        (policy and reference forward), "simpo" or "orpo" (policy forward only), then the
        loss and the streamed backward.  Hyperparameters come from the stack config."""
        if method == "dpo":
            return self.dpo_step(tok, cu, mask, self.s.beta, out)
        s = self.s
        nseq = cu.numel() - 1
        o = out if out is not None else {
            "pi": torch.empty(nseq, dtype=torch.float32, device=self.dev),
            "ref": torch.empty(nseq, dtype=torch.float32, device=self.dev),
            "loss": torch.empty(1, dtype=torch.float32, device=self.dev),
            "coeffs": torch.empty(nseq, dtype=torch.float32, device=self.dev)}
        if method in ("simpo", "orpo"):
            self.fwd(tok, cu, mask, True, True, o["pi"])
            if method == "simpo":
                check(lib().simpo_loss(self.ctx, o["pi"].data_ptr(), cu.data_ptr(), mask.data_ptr(), nseq // 2, s.beta,
                                       s.simpo_gamma, o["loss"].data_ptr(), o["coeffs"].data_ptr()), self.ctx)
            else:
                check(lib().orpo_loss(self.ctx, o["pi"].data_ptr(), cu.data_ptr(), mask.data_ptr(), nseq // 2,
                                      s.orpo_lambda, o["loss"].data_ptr(), o["coeffs"].data_ptr()), self.ctx)
        elif method == "kto":
            if self.shared_read:
                self.fwd_dpo(tok, cu, mask, o["pi"], o["ref"])
            else:
                self.fwd(tok, cu, mask, True, True, o["pi"])
                self.fwd(tok, cu, mask, False, False, o["ref"])
            check(lib().kto_loss(self.ctx, o["pi"].data_ptr(), o["ref"].data_ptr(), None, nseq, s.beta,
                                 s.kto_lambda_d, s.kto_lambda_u, o["loss"].data_ptr(), o["coeffs"].data_ptr()),
                  self.ctx)
        else:
            raise ValueError(f"unknown preference method {method!r}")
        self.bwd(o["coeffs"])
        return o

    @_stream_ordered
    def sft_step(self, tok, cu, mask, count: float, out: Optional[Dict] = None) -> Dict:
        nseq = cu.numel() - 1
        o = out if out is not None else {
            "sums": torch.empty(nseq, dtype=torch.float32, device=self.dev),
            "loss": torch.empty(1, dtype=torch.float32, device=self.dev),
            "coeffs": torch.empty(nseq, dtype=torch.float32, device=self.dev)}
        self.fwd(tok, cu, mask, True, True, o["sums"])
        check(lib().sft_loss(self.ctx, o["sums"].data_ptr(), nseq, float(count), o["loss"].data_ptr(),
                             o["coeffs"].data_ptr()), self.ctx)
        self.bwd(o["coeffs"])
        return o

    @_stream_ordered
    def train_step(self, h_tokens: torch.Tensor, h_cu: torch.Tensor, h_mask: torch.Tensor, method: str,
                   beta: float = 0.1, h_loss: Optional[torch.Tensor] = None, grads_out: Optional[torch.Tensor] = None,
                   dev_bufs: Optional[Dict] = None) -> torch.Tensor:
        """One SFT or preference step (dpo, kto, simpo, orpo) from HOST (preferably
        pinned) token, offset and mask buffers.

        Copies the batch to the device on the compute stream, runs the streamed step,
        gathers the LoRA gradients into grads_out, applies the AdamW step when
        init_optimizer was called (the gradient buffers are cleared either way), and
        copies the loss back into h_loss (fp32 [1] host).  Waits for the loss before
        returning it, like a training loop that logs every step.
        """
        d = dev_bufs if dev_bufs is not None else {}
        T, n1 = h_tokens.numel(), h_cu.numel()
        with torch.cuda.stream(self.compute):
            if "tok" not in d or d["tok"].numel() != T or d["cu"].numel() != n1:
                d["tok"] = torch.empty(T, dtype=torch.int32, device=self.dev)
                d["cu"] = torch.empty(n1, dtype=torch.int32, device=self.dev)
                d["mask"] = torch.empty(T, dtype=torch.uint8, device=self.dev)
            d["tok"].copy_(h_tokens, non_blocking=True)
            d["cu"].copy_(h_cu, non_blocking=True)
            d["mask"].copy_(h_mask, non_blocking=True)
            if method == "sft":
                o = self.sft_step(d["tok"], d["cu"], d["mask"], float(h_mask.sum().item()), d.get("out"))
            else:
                o = self.pref_step(method, d["tok"], d["cu"], d["mask"], d.get("out"))
            d["out"] = o
            if getattr(self, "opt", None) is not None:
                # gradients feed the optimizer, which clears them
                if grads_out is not None:
                    check(lib().lora_grads(self.ctx, grads_out.data_ptr(), 0), self.ctx)
                self.optimizer_step(zero_grads=True)
            else:
                check(lib().lora_grads(self.ctx, grads_out.data_ptr() if grads_out is not None else None, 1),
                      self.ctx)
            if h_loss is None:
                h_loss = torch.empty(1, dtype=torch.float32, pin_memory=True)
            h_loss.copy_(o["loss"], non_blocking=True)
        self.compute.synchronize()
        return h_loss

    @_stream_ordered
    def grads(self, zero_after: bool = False) -> torch.Tensor:
        flat = torch.empty(self.grad_numel(), dtype=torch.float32, device=self.dev)
        check(lib().lora_grads(self.ctx, flat.data_ptr(), int(zero_after)), self.ctx)
        return flat

    @_stream_ordered
    def zero_grads(self):
        check(lib().lora_grads(self.ctx, None, 1), self.ctx)

    def sync(self, timeout_ms: int = 0) -> int:
        return lib().ls_sync(self.ctx, timeout_ms)

    def stats(self, reset: bool = False) -> Dict:
        st = ls_stats_t()
        check(lib().ls_stats(self.ctx, C.byref(st), int(reset)))
        return st.as_dict()

    def close(self):
        if getattr(self, "ctx", None):
            lib().ls_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _bf16_bytes(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.uint8).numpy()
