"""Stream-K (split-tile) schedule of the fused NF4 GEMM against the oracle (GPU required).

The split schedule gives every SM the same number of k-iterations: whole 256 x 256 tiles
round-robin first, then the remaining tiles' k-iterations split evenly, the CTA holding
a tile's first iteration adding the other CTAs' fp32 partials before its epilogue.  The
cases cover one tile split over 16 CTAs (15 partials summed), ragged M and N, the LoRA
extra reduction stage landing in another CTA's share, the input-gradient (MN-major)
mode with accumulate, a round of whole tiles followed by split ones, and an exact
multiple of the SM count (whole tiles only, persistent).  Tolerance as the other GEMM
tests: normwise relative error <= 1e-2 against the fp64 oracle.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import layer_streamed_nf4_dequant_b300 as L
import oracle
import synth
from oracle import model as om

from gpu_util import DEV, bf16_dev, k, nf4_dev, rel_err, to_np

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _w(n, kk, seed, std=0.02):
    return synth.gaussian_f32((n, kk), seed, 100, n, kk, std=std)


def _deq(w):
    c, a = oracle.nf4_quantize(w)
    return oracle.nf4_dequantize(c, a)


_WS = {}


def _ws():
    if "ws" not in _WS:
        n = int(L.lib().lsk_nf4_gemm_workspace_bytes())
        _WS["ws"] = torch.zeros(n, dtype=torch.uint8, device=DEV)
    return _WS["ws"]


def _sk(mode, x, M, p, a, N, K, ext_a, ext_b, ext_k, epi, out, ldo, res, split, pair_rows=0):
    ws = _ws()
    red = K if mode == 0 else N
    k("lsk_nf4_gemm_sk", mode, x, red, M, p, a, N, K, ext_a, ext_b, ext_k, epi, out, ldo, res,
      (ldo if res is not None else 0), 0, 0, split, pair_rows, ws, ws.numel())


def _check_device_error():
    e = ctypes.c_int32(0)
    assert L.lib().lsk_device_error(ctypes.byref(e), 1) == 0
    assert e.value == 0, f"device error word {e.value}"


FWD_CASES = [
    # (M, N, K, sampled rows or None)
    (256, 256, 4096, None),        # one tile, 64 iterations over 16 CTAs
    (513, 768, 1024, None),        # ragged M: 3 x 3 tiles
    (300, 320, 640, None),         # ragged M and N (last column tile 64 wide)
    (1024, 4096, 4096, [0, 1, 255, 256, 700, 1023]),   # 64 tiles over the SMs
    (2048, 9728, 256, [0, 77, 1024, 2047]),            # 304 tiles: one whole round, then split
    (256, 148 * 256, 128, [0, 100, 255]),              # 148 tiles: whole, persistent
]


@pytest.mark.parametrize("M,N,K,rows", FWD_CASES)
def test_split_fwd_bf16_and_residual(M, N, K, rows):
    x = synth.gaussian((M, K), 31, M, K)
    w = _w(N, K, seed=32)
    res = synth.gaussian((M, N), 33, M, N)
    p, a, _, _ = nf4_dev(w)
    wd = _deq(w)
    xd, rd = bf16_dev(x), bf16_dev(res)
    sel = np.arange(M) if rows is None else np.array(rows)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    _sk(0, xd, M, p, a, N, K, None, None, 0, 0, out, N, None, 1)
    torch.cuda.synchronize()
    got = to_np(out)[sel]
    want = om.linear(om.t64(x[sel]), om.t64(wd)).numpy()
    assert rel_err(got, want) <= TOL
    # deterministic: the partials are added in a fixed order
    out2 = torch.empty_like(out)
    _sk(0, xd, M, p, a, N, K, None, None, 0, 0, out2, N, None, 1)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
    _sk(0, xd, M, p, a, N, K, None, None, 0, 0, out, N, rd, 1)
    torch.cuda.synchronize()
    want = om.linear(om.t64(x[sel]), om.t64(wd), residual=om.t64(res[sel])).numpy()
    assert rel_err(to_np(out)[sel], want) <= TOL
    _check_device_error()


DX_CASES = [
    # (M, N, K): dX [M, K] = dY [M, N] . deq(W) [N, K]
    (512, 4096, 1024),     # 8 tiles, 64 iterations each, split over the SMs
    (384, 2048, 768),      # ragged M
    (256, 14336, 512),     # long reduction: 2 tiles x 224 iterations
]


@pytest.mark.parametrize("M,N,K", DX_CASES)
def test_split_dx_f32_and_accumulate(M, N, K):
    dy = synth.gaussian((M, N), 34, M, N)
    w = _w(N, K, seed=35)
    p, a, _, _ = nf4_dev(w)
    wd = _deq(w)
    out = torch.empty((M, K), dtype=torch.float32, device=DEV)
    dyd = bf16_dev(dy)
    _sk(1, dyd, M, p, a, N, K, None, None, 0, 1, out, K, None, 1)
    torch.cuda.synchronize()
    want = dy.astype(np.float64) @ wd.astype(np.float64)
    assert rel_err(to_np(out), want) <= TOL
    _sk(1, dyd, M, p, a, N, K, None, None, 0, 2, out, K, None, 1)
    torch.cuda.synchronize()
    assert rel_err(to_np(out), 2 * want) <= TOL
    _check_device_error()


def test_split_lora_extra_stage_in_another_share():
    """K = 1024 plus the LoRA stage: 17 iterations of one tile over 4 CTAs, so the extra
    reduction stage is the last CTA's partial; forward and input gradient."""
    T, Kd, Nd, r, s = 256, 1024, 256, 16, 2.0
    x = synth.gaussian((T, Kd), 36, 1)
    w = _w(Nd, Kd, seed=37)
    a_ = synth.gaussian((r, Kd), 36, 2, std=0.05)
    b_ = synth.gaussian((Nd, r), 36, 3, std=0.05)
    dy = synth.gaussian((T, Nd), 36, 4)
    p, am, _, _ = nf4_dev(w)
    xd, ad, bd, dyd = bf16_dev(x), bf16_dev(a_), bf16_dev(b_), bf16_dev(dy)
    u_ext = torch.empty((T, 64), dtype=torch.bfloat16, device=DEV)
    ext_b = torch.empty((Nd, 64), dtype=torch.bfloat16, device=DEV)
    k("lsk_lora_down", xd, Kd, ad, None, r, Kd, s, u_ext, T)
    k("lsk_build_ext_fwd", bd, 0, Nd, None, 0, 0, r, Nd, ext_b)
    y = torch.empty((T, Nd), dtype=torch.bfloat16, device=DEV)
    _sk(0, xd, T, p, am, Nd, Kd, u_ext, ext_b, 16, 0, y, Nd, None, 1)
    du = torch.empty((T, 32), dtype=torch.float32, device=DEV)
    du_ext = torch.empty((T, 64), dtype=torch.bfloat16, device=DEV)
    k("lsk_lora_du", dyd, Nd, 0, Nd, bd, 0, 0, None, r, s, du, du_ext, T)
    ext_a = torch.empty((Kd, 64), dtype=torch.bfloat16, device=DEV)
    k("lsk_build_ext_bwd", ad, None, r, Kd, ext_a)
    dx = torch.empty((T, Kd), dtype=torch.float32, device=DEV)
    _sk(1, dyd, T, p, am, Nd, Kd, du_ext, ext_a, 16, 1, dx, Kd, None, 1)
    ref = om.lora_linear_step(x, _deq(w), a_, b_, s, dy)
    torch.cuda.synchronize()
    assert rel_err(to_np(y), ref["y"].numpy()) <= TOL
    assert rel_err(to_np(dx), ref["dx"].numpy()) <= TOL
    _check_device_error()


def test_split_matches_whole_tiles_and_auto():
    """Split, whole-tile and cost-model schedules of the same product agree to fp32
    summation-order differences."""
    M, N, K = 1024, 6144, 4096
    x = synth.gaussian((M, K), 38, 1)
    w = _w(N, K, seed=39)
    p, a, _, _ = nf4_dev(w)
    xd = bf16_dev(x)
    outs = []
    for split in (1, -1, 0):
        o = torch.empty((M, N), dtype=torch.float32, device=DEV)
        _sk(0, xd, M, p, a, N, K, None, None, 0, 1, o, N, None, split)
        outs.append(o)
    torch.cuda.synchronize()
    ref = outs[1].double()
    scale = ref.abs().max().item()
    for o in (outs[0], outs[2]):
        assert (o.double() - ref).abs().max().item() <= 1e-5 * scale
    _check_device_error()


@pytest.mark.parametrize("T,N,K,ext", [(1024, 6144, 4096, 0), (300, 640, 1024, 16)])
def test_paired_halves_round_identically(T, N, K, ext):
    """The shared-read forward's batch [X; X] (pair_rows = T) on the split schedule: both
    halves bit-identical (row r and row T + r share a CTA and its k-splits), and within
    the tolerance of the oracle; T = 300 leaves a ragged last 128-row block."""
    x = synth.gaussian((T, K), 42, T, K)
    w = _w(N, K, seed=43)
    res = synth.gaussian((T, N), 44, T, N)
    p, a, _, _ = nf4_dev(w)
    wd = _deq(w)
    x2, r2 = bf16_dev(np.concatenate([x, x])), bf16_dev(np.concatenate([res, res]))
    ext_a = ext_b = None
    if ext:
        u = synth.gaussian((T, 64), 45, T) * (np.arange(64) < ext)
        b = synth.gaussian((N, 64), 46, N) * (np.arange(64) < ext) * 0.05
        ext_a, ext_b = bf16_dev(np.concatenate([u, u])), bf16_dev(b)
    out = torch.empty((2 * T, N), dtype=torch.bfloat16, device=DEV)
    _sk(0, x2, 2 * T, p, a, N, K, ext_a, ext_b, ext, 0, out, N, r2, 1, pair_rows=T)
    torch.cuda.synchronize()
    assert torch.equal(out[:T], out[T:])
    lora = None
    if ext:
        lora = (om.t64(np.asarray(to_np(ext_a[:T]))), om.t64(np.asarray(to_np(ext_b))))
    want = om.linear(om.t64(x), om.t64(wd), lora=lora, residual=om.t64(res)).numpy()
    assert rel_err(to_np(out[:T]), want) <= TOL
    _check_device_error()


@pytest.mark.parametrize("T,N,K,ext", [(1024, 6144, 4096, 32), (1024, 28672, 4096, 0), (1024, 4096, 14336, 0),
                                       (300, 640, 1024, 16)])
def test_paired_halves_differ_and_match_whole_tiles(T, N, K, ext):
    """A paired batch [X; Y] with different halves (the shared-read forward's policy and
    reference rows once the adapter has moved them apart): each half must be its own
    product.  Against whole tiles of the same batch the paired split differs only in
    fp32 summation order; against the oracle each half is within the product bound."""
    x = synth.gaussian((2 * T, K), 47, T, K)
    w = _w(N, K, seed=48)
    p, a, _, _ = nf4_dev(w)
    wd = _deq(w)
    xd = bf16_dev(x)
    ext_a = ext_b = None
    u = b = None
    if ext:
        u = synth.gaussian((2 * T, 64), 49, T) * (np.arange(64) < ext)
        b = synth.gaussian((N, 64), 50, N) * (np.arange(64) < ext) * 0.05
        ext_a, ext_b = bf16_dev(u), bf16_dev(b)
    paired = torch.empty((2 * T, N), dtype=torch.float32, device=DEV)
    whole = torch.empty((2 * T, N), dtype=torch.float32, device=DEV)
    _sk(0, xd, 2 * T, p, a, N, K, ext_a, ext_b, ext, 1, paired, N, None, 1, pair_rows=T)
    _sk(0, xd, 2 * T, p, a, N, K, ext_a, ext_b, ext, 1, whole, N, None, -1)
    torch.cuda.synchronize()
    ref = whole.double()
    scale = ref.abs().max().item()
    # two fp32 summation orders of K products: their difference walks like sqrt(K) unit
    # roundoffs of the running sum (8x room)
    assert (paired.double() - ref).abs().max().item() <= 8 * math.sqrt(K) * 2.0 ** -24 * scale
    rows = np.array([0, 1, T - 1, T, T + 1, 2 * T - 1, T // 2, T + T // 2])
    xr = bf16_dev(x[rows]).float().cpu().numpy()
    lora = None
    if ext:
        lora = (om.t64(to_np(ext_a)[rows]), om.t64(to_np(ext_b)))
    want = om.linear(om.t64(xr), om.t64(wd), lora=lora).numpy()
    assert rel_err(to_np(paired)[rows], want) <= TOL
    _check_device_error()


@pytest.mark.parametrize("mode,split", [(0, 1), (0, -1), (1, 1), (1, -1)])
def test_one_hot_rows_reproduce_the_dequant_exactly(mode, split):
    """With one-hot activation rows every output of the fused product is a single
    dequantised weight (times 1, plus exact zeros), so the GEMM's in-shared-memory dequant
    must equal the definition bit for bit: forward out[m, n] = deq(W)[n, m], input
    gradient out[m, k] = deq(W)[m, k].  N(0, 0.02) weights use all 16 codes, so both
    halves of the byte tables and the >= 8 mask are exercised, on whole and split tiles."""
    N, K = 512, 1024
    w = _w(N, K, seed=51)
    p, a, _, _ = nf4_dev(w)
    wd = _deq(w)
    M = K if mode == 0 else N
    red = K if mode == 0 else N
    x = torch.eye(M, red, dtype=torch.bfloat16, device=DEV).contiguous()
    outc = N if mode == 0 else K
    out = torch.empty((M, outc), dtype=torch.float32, device=DEV)
    _sk(mode, x, M, p, a, N, K, None, None, 0, 1, out, outc, None, split)
    torch.cuda.synchronize()
    want = torch.from_numpy(np.ascontiguousarray(wd.T if mode == 0 else wd))
    assert torch.equal(out.cpu(), want)
    _check_device_error()


def test_split_rejects_small_workspace():
    ws = _ws()
    x = torch.zeros((256, 256), dtype=torch.bfloat16, device=DEV)
    w = _w(256, 256, seed=40)
    p, a, _, _ = nf4_dev(w)
    out = torch.empty((256, 256), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(L.LSError):
        k("lsk_nf4_gemm_sk", 0, x, 256, 256, p, a, 256, 256, None, None, 0, 0, out, 256, None, 0, 0, 0, 1, 0,
          ws, ws.numel() - 1)
