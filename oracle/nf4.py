"""NF4 block quantisation and dequantisation — oracle (test infrastructure only).

The pages say only that the streamed frozen base is optionally quantised to NF4,
shrinking the store about fourfold (Soup: Fine-Tune an 8B Model on a 4 GB GPU,
"The Core Idea: Layer Streaming" and its soup.yaml listing, "quantization: 4bit
# NF4").  The format itself is the one QLoRA published (Dettmers et al. 2023,
"QLoRA: Efficient Finetuning of Quantized LLMs", Sec. 3 "4-bit NormalFloat
Quantization" and Appendix E's table of NF4 values): 16 code values, one absmax
scale per block of 64 consecutive weights.

Readings taken where the pages are silent:
  * absmax is stored as fp32, with no double quantisation;
  * the code of w is the table entry nearest to w / absmax, the fp32 quotient,
    with distance |w/absmax - q_j| in fp32 and ties going to the lower index;
    an all-zero block (absmax = 0) gets code 7, the exact zero;
  * two codes per byte, element 2i in the high nibble and 2i+1 in the low one;
  * dequantisation is one fp32 multiply q[c] * absmax, rounded once to bf16
    (round to nearest even).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

BLOCK = 64

# QLoRA Appendix E: the 16 NormalFloat-4 values (ascending, q[7] == 0 exactly).
NF4_TABLE = np.array([
    -1.0, -0.6961928009986877, -0.5250730514526367, -0.39491748809814453,
    -0.28444138169288635, -0.18477343022823334, -0.09105003625154495, 0.0,
    0.07958029955625534, 0.16093020814657211, 0.24611230194568634, 0.33791524171829224,
    0.44070982933044434, 0.5626170039176941, 0.7229568362236023, 1.0], dtype=np.float32)


def bf16_round_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returns fp32 holding them.

    Written out on the bit pattern: keep the top 16 bits after adding half an ulp
    of the kept part, plus one when the kept part is odd (round half to even).
    NaNs are passed through as quiet NaNs.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)).astype(np.uint32)
    out = r.view(np.float32).copy()
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.float32(np.nan)
    return out


def nf4_quantize(w: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Quantise fp32 W [N, K] (K % 64 == 0) to codes uint8 [N, K] and absmax fp32 [N, K/64].

    Per 64-element block of a row: absmax = max |w_i|; code_i = argmin_j |w_i/absmax - q_j|.
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    if k % BLOCK:
        raise ValueError("K must be a multiple of 64")
    blocks = w.reshape(n, k // BLOCK, BLOCK)
    absmax = np.abs(blocks).max(axis=2).astype(np.float32)
    codes = np.empty((n, k // BLOCK, BLOCK), np.uint8)

    def rows(r0, r1):
        with np.errstate(invalid="ignore", divide="ignore"):
            x = blocks[r0:r1] / absmax[r0:r1, :, None]          # fp32 quotient
        # argmin_j |x - q_j| as a running minimum over j; strict '<' keeps the lower index on ties
        best = np.abs(x - NF4_TABLE[0])
        c = np.zeros(x.shape, np.uint8)
        d = np.empty_like(x)
        better = np.empty(x.shape, bool)
        for j in range(1, 16):
            np.subtract(x, NF4_TABLE[j], out=d)
            np.abs(d, out=d)
            np.less(d, best, out=better)
            np.copyto(best, d, where=better)
            np.copyto(c, np.uint8(j), where=better)
        c[np.broadcast_to(absmax[r0:r1, :, None] == 0, c.shape)] = 7
        codes[r0:r1] = c

    step = max(1, (1 << 20) // k)
    spans = [(r0, min(n, r0 + step)) for r0 in range(0, n, step)]
    if len(spans) > 1:
        with ThreadPoolExecutor(min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(lambda sp: rows(*sp), spans))
    else:
        rows(0, n)
    return codes.reshape(n, k), absmax


def nf4_pack(codes: np.ndarray) -> np.ndarray:
    """Pack codes uint8 [N, K] into bytes [N, K/2]: element 2i high nibble, 2i+1 low nibble."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    return ((c[:, 0::2] << 4) | c[:, 1::2]).astype(np.uint8)


def nf4_unpack(packed: np.ndarray) -> np.ndarray:
    """Inverse of nf4_pack."""
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    n, kh = p.shape
    c = np.empty((n, kh * 2), np.uint8)
    c[:, 0::2] = p >> 4
    c[:, 1::2] = p & 0xF
    return c


def nf4_dequantize(codes: np.ndarray, absmax: np.ndarray) -> np.ndarray:
    """Dequantise codes [N, K] with absmax [N, K/64]: bf16_RNE(fp32(q[c]) * absmax), as fp32."""
    n, k = codes.shape
    q = NF4_TABLE[codes].reshape(n, k // BLOCK, BLOCK)
    prod = (q * absmax[:, :, None].astype(np.float32)).astype(np.float32)  # one fp32 multiply
    return bf16_round_f32(prod.reshape(n, k))
