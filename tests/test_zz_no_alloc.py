"""The allocation-free LoRA outer-product entry point (GPU required).

lsk_lora_outer_noalloc serves callers that cannot allocate device memory (code
running inside another framework's memory pool, or on paths that must not take
cudaMalloc's implicit synchronisation): it keeps its partial sums in a fixed array
inside the library instead of caller scratch.  These tests call it through the C ABI
and check it against the scratch-taking lsk_lora_outer on the same inputs, twice in a
row with different inputs (the shared array keeps the previous call's contents).  Both
run the same kernels over the same chunks in the same order, so the results must be
equal bit for bit.  An oversized request must be refused before anything is launched.
This file is collected last so that a failure here cannot hide any other test.
"""
import math

import numpy as np
import pytest
import torch

import layer_streamed_nf4_dequant_b300 as L
import synth

from gpu_util import DEV, bf16_dev, rel_err, stream, to_np

pytestmark = pytest.mark.gpu

TOL = 1e-2     # the normwise bound the kernel tests use for products
MAX_FLOATS = 2097152


def _outer_both(X, ncols, U_f32, U_bf16, ldu, r, T, layout, accumulate, rpc, seed):
    nch = math.ceil(T / rpc)
    scratch = torch.empty(nch * ncols * 16, dtype=torch.float32, device=DEV)
    shape = (ncols, r) if layout == 0 else (r, ncols)
    init = torch.from_numpy(synth.gaussian_f32(shape, seed, 7)).to(DEV)
    want, got = init.clone(), init.clone()
    L.call("lsk_lora_outer", X, ncols, ncols, U_f32, U_bf16, ldu, r, T, layout, accumulate, scratch, rpc, want,
           stream())
    L.call("lsk_lora_outer_noalloc", X, ncols, ncols, U_f32, U_bf16, ldu, r, T, layout, accumulate, rpc, got,
           stream())
    torch.cuda.synchronize()
    return want, got


def test_noalloc_outer_matches_scratch_version_two_calls_in_a_row():
    # call 1: dA shape (r x ncols) from fp32 u, 8B width, 1024 tokens
    T1, n1, r = 1024, 4096, 16
    X1 = bf16_dev(synth.gaussian((T1, n1), 40, 1))
    U1 = torch.from_numpy(synth.gaussian_f32((T1, 32), 41, 1)).to(DEV)
    want1, got1 = _outer_both(X1, n1, U1, None, 32, r, T1, 1, 0, 128, 42)
    assert torch.equal(got1, want1)
    # call 2 right after: dB shape (ncols x r) from bf16 u, ragged T, accumulate onto
    # existing values -- a smaller problem, so stale partials of call 1 sit beyond it
    T2, n2, r2 = 300, 1024, 8
    X2 = bf16_dev(synth.gaussian((T2, n2), 43, 2))
    U2 = bf16_dev(synth.gaussian((T2, 64), 44, 2))
    want2, got2 = _outer_both(X2, n2, None, U2, 64, r2, T2, 0, 1, 128, 45)
    assert torch.equal(got2, want2)
    # and against a plain fp64 product, to be sure both are the real thing
    x = to_np(X2)
    u = to_np(U2)[:, :r2]
    init = synth.gaussian_f32((n2, r2), 45, 7).astype(np.float64)
    assert rel_err(to_np(got2), init + x.T @ u) <= TOL


def test_noalloc_outer_refuses_sizes_beyond_its_array():
    T, ncols, r, rpc = 8192, 8192, 16, 128   # 64 chunks x 8192 x 16 floats > 2^21
    assert math.ceil(T / rpc) * ncols * 16 > MAX_FLOATS
    X = torch.zeros((T, ncols), dtype=torch.bfloat16, device=DEV)
    U = torch.zeros((T, 32), dtype=torch.float32, device=DEV)
    out = torch.zeros((r, ncols), dtype=torch.float32, device=DEV)
    rc = L.lib().lsk_lora_outer_noalloc(X.data_ptr(), ncols, ncols, U.data_ptr(), None, 32, r, T, 1, 0, rpc,
                                        out.data_ptr(), stream())
    assert rc == L.LS_ERR_ARG
    assert "more than the fixed" in L.last_error()


def test_noalloc_outer_compact_u():
    """U stored compactly ([T, r], ldu = r < 16): only its r columns are read."""
    T, ncols, r = 200, 512, 8
    X = bf16_dev(synth.gaussian((T, ncols), 46, 3))
    U = torch.from_numpy(synth.gaussian_f32((T, r), 47, 3)).to(DEV)
    want, got = _outer_both(X, ncols, U, None, r, r, T, 1, 0, 64, 48)
    assert torch.equal(got, want)
    assert rel_err(to_np(got), to_np(U).T @ to_np(X)) <= TOL
