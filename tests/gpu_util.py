"""Helpers for the GPU parity tests: device tensors, comparisons, C-ABI calls."""
import numpy as np
import torch

import layer_streamed_nf4_dequant_b300 as L

DEV = torch.device("cuda:0")


def stream():
    return torch.cuda.current_stream().cuda_stream


def bf16_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).to(DEV)


def as_u16(t: torch.Tensor) -> int:
    return t.data_ptr()


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_err(got, want) -> float:
    """Normwise relative error: max|got - want| / max|want|."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    den = np.abs(want).max()
    return float(np.abs(got - want).max() / (den if den > 0 else 1.0))


def nf4_dev(w: np.ndarray):
    """Quantise with the library's host quantiser; device packed + absmax tensors."""
    pk, am = L.quantize_host(w)
    return torch.from_numpy(pk).to(DEV), torch.from_numpy(am).to(DEV), pk, am


def k(name, *args):
    """Call a kernel-level entry point on the current stream."""
    return L.call(name, *args, stream())
