"""Kernel-level parity of the CUDA path against the oracle (GPU required).

Tolerances: NF4 dequantisation bit-exact; matrix products and layer pieces
normwise relative error <= 1e-2 (max|gpu - oracle| / max|oracle|); logprobs
absolute error <= 2e-2.
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

from gpu_util import DEV, bf16_dev, k, nf4_dev, rel_err, stream, to_np

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _w(n, kk, seed, std=0.02):
    return synth.gaussian_f32((n, kk), seed, 100, n, kk, std=std)


def _oracle_deq(w):
    c, a = oracle.nf4_quantize(w)
    return oracle.nf4_dequantize(c, a)


# ------------------------------------------------------------------ dequant

@pytest.mark.parametrize("shape", [(64, 64), (256, 896), (1000, 4864), (14336, 4096)])
def test_dequant_bit_exact(shape):
    w = _w(*shape, seed=1)
    p, a, pk, am = nf4_dev(w)
    out = torch.empty(shape, dtype=torch.bfloat16, device=DEV)
    k("lsk_nf4_dequant", p, a, shape[0], shape[1], out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    np.testing.assert_array_equal(got, _oracle_deq(w))


# ------------------------------------------------------------------ fused GEMM

GEMM_CASES = [
    # (M, N, K, force_bn, force_nacc)
    (64, 256, 256, 0, 0),          # the single-linear shape
    (512, 1152, 896, 0, 0),        # fused q/k/v of the 896-wide layer (ragged N for 256 tiles)
    (200, 384, 640, 128, 1),       # ragged M, several K stages
    (300, 512, 1024, 256, 1),
    (700, 640, 512, 128, 2),
    (513, 768, 384, 256, 2),
]


@pytest.mark.parametrize("M,N,K,bn,nacc", GEMM_CASES)
def test_gemm_fwd_and_residual(M, N, K, bn, nacc):
    x = synth.gaussian((M, K), 3, M, K)
    w = _w(N, K, seed=2)
    res = synth.gaussian((M, N), 4, M, N)
    p, a, _, _ = nf4_dev(w)
    wd = _oracle_deq(w)
    xd = bf16_dev(x)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    k("lsk_nf4_gemm", 0, xd, K, M, p, a, N, K, None, None, 0, 0, out, N, None, 0, bn, nacc)
    want = om.linear(om.t64(x), om.t64(wd)).numpy()
    torch.cuda.synchronize()
    assert rel_err(to_np(out), want) <= TOL
    rd = bf16_dev(res)
    k("lsk_nf4_gemm", 0, xd, K, M, p, a, N, K, None, None, 0, 0, out, N, rd, N, bn, nacc)
    want = om.linear(om.t64(x), om.t64(wd), residual=om.t64(res)).numpy()
    torch.cuda.synchronize()
    assert rel_err(to_np(out), want) <= TOL


@pytest.mark.parametrize("bn,nacc", [(128, 1), (256, 2)])
def test_gemm_fwd_into_a_column_window_of_a_wider_output(bn, nacc):
    """bf16 outputs leave through 32-row x 64-column tensor-store boxes clipped at the
    product's own rows and columns: written into columns 8 .. 8 + N of a 512-wide buffer
    (row pitch 512, ragged M and N), the product equals the compact one bit for bit and
    every other column keeps its old value."""
    M, N, K = 300, 384, 256
    x = synth.gaussian((M, K), 31, M, K)
    w = _w(N, K, seed=32)
    p, a, _, _ = nf4_dev(w)
    xd = bf16_dev(x)
    buf = torch.full((M, 512), 7.0, dtype=torch.bfloat16, device=DEV)
    compact = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    k("lsk_nf4_gemm", 0, xd, K, M, p, a, N, K, None, None, 0, 0, buf[:, 8:8 + N], 512, None, 0, bn, nacc)
    k("lsk_nf4_gemm", 0, xd, K, M, p, a, N, K, None, None, 0, 0, compact, N, None, 0, bn, nacc)
    want = om.linear(om.t64(x), om.t64(_oracle_deq(w))).numpy()
    torch.cuda.synchronize()
    assert torch.equal(buf[:, 8:8 + N], compact)
    assert bool((buf[:, :8] == 7.0).all()) and bool((buf[:, 8 + N:] == 7.0).all())
    assert rel_err(to_np(compact), want) <= TOL


@pytest.mark.parametrize("M,N,K,bn,nacc", GEMM_CASES)
def test_gemm_dx(M, N, K, bn, nacc):
    dy = synth.gaussian((M, N), 5, M, N)
    w = _w(N, K, seed=6)
    p, a, _, _ = nf4_dev(w)
    wd = _oracle_deq(w)
    out = torch.empty((M, K), dtype=torch.float32, device=DEV)
    k("lsk_nf4_gemm", 1, bf16_dev(dy), N, M, p, a, N, K, None, None, 0, 1, out, K, None, 0, bn, nacc)
    want = dy.astype(np.float64) @ wd.astype(np.float64)
    torch.cuda.synchronize()
    assert rel_err(to_np(out), want) <= TOL
    # accumulate mode adds onto what is there
    k("lsk_nf4_gemm", 1, bf16_dev(dy), N, M, p, a, N, K, None, None, 0, 2, out, K, None, 0, bn, nacc)
    torch.cuda.synchronize()
    assert rel_err(to_np(out), 2 * want) <= TOL


def test_gemm_full_size_sampled_rows():
    """8B-shape fused gate/up product (T=1024, N=28672, K=4096); 8 sampled rows vs the oracle."""
    M, N, K = 1024, 2 * 14336, 4096
    x = synth.gaussian((M, K), 7, 1)
    w = _w(N, K, seed=8)
    p, a, _, _ = nf4_dev(w)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    k("lsk_nf4_gemm", 0, bf16_dev(x), K, M, p, a, N, K, None, None, 0, 0, out, N, None, 0, 0, 0)
    rows = np.array([0, 1, 127, 128, 255, 511, 777, 1023])
    wd = _oracle_deq(w)
    want = om.linear(om.t64(x[rows]), om.t64(wd)).numpy()
    torch.cuda.synchronize()
    assert rel_err(to_np(out[rows]), want) <= TOL


def test_lora_linear_single_shape_fwd_bwd():
    """The single NF4 LoRA linear (d_in = d_out = 256, 64 tokens, r 8, alpha 16) fwd + bwd."""
    cfg = synth.LINEAR_256
    T, Kd, Nd, r, s = cfg["tokens"], cfg["d_in"], cfg["d_out"], cfg["r"], cfg["alpha"] / cfg["r"]
    x = synth.gaussian((T, Kd), 0, 1)
    w = _w(Nd, Kd, seed=0)
    a = synth.gaussian((r, Kd), 0, 2, std=0.01)
    b = synth.gaussian((Nd, r), 0, 3, std=0.01)
    dy = synth.gaussian((T, Nd), 0, 4)
    p, am, _, _ = nf4_dev(w)
    xd, ad, bd, dyd = bf16_dev(x), bf16_dev(a), bf16_dev(b), bf16_dev(dy)
    u_ext = torch.empty((T, 64), dtype=torch.bfloat16, device=DEV)
    ext_b = torch.empty((Nd, 64), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((T, Nd), dtype=torch.bfloat16, device=DEV)
    k("lsk_lora_down", xd, Kd, ad, None, r, Kd, s, u_ext, T)
    k("lsk_build_ext_fwd", bd, 0, Nd, None, 0, 0, r, Nd, ext_b)
    k("lsk_nf4_gemm", 0, xd, Kd, T, p, am, Nd, Kd, u_ext, ext_b, 16, 0, y, Nd, None, 0, 0, 0)
    # backward: du = s dY B, dB = dY^T u, dA = (s du)^T x, dX = dY W + (s du) A
    du = torch.empty((T, 32), dtype=torch.float32, device=DEV)
    du_ext = torch.empty((T, 64), dtype=torch.bfloat16, device=DEV)
    k("lsk_lora_du", dyd, Nd, 0, Nd, bd, 0, 0, None, r, s, du, du_ext, T)
    scratch = torch.empty(4 * 256 * 16, dtype=torch.float32, device=DEV)
    db = torch.zeros((Nd, r), dtype=torch.float32, device=DEV)
    da = torch.zeros((r, Kd), dtype=torch.float32, device=DEV)
    k("lsk_lora_outer", dyd, Nd, Nd, None, u_ext, 64, r, T, 0, 0, scratch, 16, db)
    k("lsk_lora_outer", xd, Kd, Kd, du, None, 32, r, T, 1, 0, scratch, 16, da)
    ext_a = torch.empty((Kd, 64), dtype=torch.bfloat16, device=DEV)
    k("lsk_build_ext_bwd", ad, None, r, Kd, ext_a)
    dx = torch.empty((T, Kd), dtype=torch.float32, device=DEV)
    k("lsk_nf4_gemm", 1, dyd, Nd, T, p, am, Nd, Kd, du_ext, ext_a, 16, 1, dx, Kd, None, 0, 0, 0)
    ref = om.lora_linear_step(x, _oracle_deq(w), a, b, s, dy)
    torch.cuda.synchronize()
    assert rel_err(to_np(y), ref["y"].numpy()) <= TOL
    assert rel_err(to_np(dx), ref["dx"].numpy()) <= TOL
    assert rel_err(to_np(da), ref["da"].numpy()) <= TOL
    assert rel_err(to_np(db), ref["db"].numpy()) <= TOL
    # B = 0: the extra stage adds exact zeros -> bit-identical to the base product
    y0 = torch.empty_like(y)
    yb = torch.empty_like(y)
    k("lsk_build_ext_fwd", torch.zeros_like(bd), 0, Nd, None, 0, 0, r, Nd, ext_b)
    k("lsk_nf4_gemm", 0, xd, Kd, T, p, am, Nd, Kd, u_ext, ext_b, 16, 0, y0, Nd, None, 0, 0, 0)
    k("lsk_nf4_gemm", 0, xd, Kd, T, p, am, Nd, Kd, None, None, 0, 0, yb, Nd, None, 0, 0, 0)
    torch.cuda.synchronize()
    assert torch.equal(y0, yb)


# ------------------------------------------------------------------ embedding gather

def test_embed_gather_rows_and_out_of_range_ids():
    """Rows of the NF4 embedding bit-exact against the oracle's dequantisation; ids V and
    -1 give zero rows and set the device error word (checked before any access with the
    id), and the context stays usable."""
    V, H = 300, 256
    w = _w(V, H, seed=41)
    p, a, _, _ = nf4_dev(w)
    wd = _oracle_deq(w)
    ids = np.array([0, 299, 7, 300, -1, 150], np.int32)
    tok = torch.from_numpy(ids).to(DEV)
    x = torch.full((len(ids), H), 1.0, dtype=torch.bfloat16, device=DEV)
    e = ctypes.c_int32(0)
    assert L.lib().lsk_device_error(ctypes.byref(e), 1) == 0
    k("lsk_embed_gather", tok, p, a, V, x, len(ids), H)
    torch.cuda.synchronize()
    got = x.float().cpu().numpy()
    for i in (0, 1, 2, 5):
        np.testing.assert_array_equal(got[i], wd[ids[i]])
    assert not got[3].any() and not got[4].any()
    assert L.lib().lsk_device_error(ctypes.byref(e), 1) == 0
    assert e.value == 2   # bad argument seen by a kernel
    k("lsk_embed_gather", tok[:3], p, a, V, x, 3, H)
    torch.cuda.synchronize()
    assert L.lib().lsk_device_error(ctypes.byref(e), 1) == 0 and e.value == 0


# ------------------------------------------------------------------ bounded waits

def test_bounded_wait_runs_out_and_context_stays_usable():
    """A wait on a flag that nothing sets ends after its limit with status 1 and the
    device error word 1 (wait timeout); a flag already set is seen at once (status 0,
    no error); later kernels run normally on the same context."""
    flag = torch.zeros(4, dtype=torch.int32, device=DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    e = ctypes.c_int32(0)
    assert L.lib().lsk_device_error(ctypes.byref(e), 1) == 0
    k("lsk_wait_flag", flag, 1, 20_000_000, status)          # 20 ms, nobody sets it
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert L.lib().lsk_device_error(ctypes.byref(e), 1) == 0 and e.value == 1
    flag.fill_(7)
    status.fill_(-1)
    k("lsk_wait_flag", flag, 7, 20_000_000, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert L.lib().lsk_device_error(ctypes.byref(e), 1) == 0 and e.value == 0
    assert L.lib().lsk_wait_flag(flag.data_ptr() + 2, 0, 1000, status.data_ptr(), stream()) == L.LS_ERR_ARG
    x = torch.ones(1024, device=DEV)
    assert float((x * 2).sum()) == 2048.0


# ------------------------------------------------------------------ norms, rope, swiglu

@pytest.mark.parametrize("T,H", [(5, 64), (512, 896), (1024, 4096), (37, 5120)])
def test_rmsnorm_fwd_bwd(T, H):
    x = synth.gaussian((T, H), 9, T, H, std=3.0)
    w = synth.gaussian((H,), 10, H) + 1.0
    w = synth.to_bf16_values(w)
    dy = synth.gaussian_f32((T, H), 11, T)
    xd, wd = bf16_dev(x), bf16_dev(w)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    rstd = torch.empty(T, dtype=torch.float32, device=DEV)
    k("lsk_rmsnorm_fwd", xd, wd, y, rstd, T, H, 1e-6)
    X = om.t64(x).requires_grad_(True)
    yo = om.rmsnorm(X, om.t64(w), 1e-6)
    (yo * om.t64(dy)).sum().backward()
    dx = torch.zeros((T, H), dtype=torch.float32, device=DEV)
    dxb = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    k("lsk_rmsnorm_bwd", torch.from_numpy(dy).to(DEV), xd, rstd, wd, dx, dxb, T, H, 0)
    torch.cuda.synchronize()
    assert rel_err(to_np(y), yo.detach().numpy()) <= TOL
    assert rel_err(to_np(dx), X.grad.numpy()) <= TOL
    assert torch.equal(dxb, dx.to(torch.bfloat16))


def _rope_tabs(maxp, hd, theta):
    c = np.empty((maxp, hd // 2), np.float32)
    s = np.empty_like(c)
    L.check(L.lib().ls_rope_table(c.ctypes.data, s.ctypes.data, maxp, hd, theta))
    return torch.from_numpy(c).to(DEV), torch.from_numpy(s).to(DEV)


@pytest.mark.parametrize("hd,nh,nkv", [(64, 14, 2), (128, 32, 8)])
def test_rope_fwd_bwd(hd, nh, nkv):
    T = 300
    cu = [0, 100, 300]
    pos = np.concatenate([np.arange(100), np.arange(200)]).astype(np.int32)
    ncols = (nh + 2 * nkv) * hd
    qkv = synth.gaussian((T, ncols), 12, hd)
    ct, st = _rope_tabs(256, hd, 1e6)
    d = bf16_dev(qkv)
    posd = torch.from_numpy(pos).to(DEV)
    k("lsk_rope_fwd", d, ncols, posd, ct, st, T, nh + nkv, hd)
    P = torch.from_numpy(pos.astype(np.int64))
    q = om.rope(om.t64(qkv[:, :nh * hd]).view(T, nh, hd), P, 1e6).reshape(T, -1).numpy()
    kk = om.rope(om.t64(qkv[:, nh * hd:(nh + nkv) * hd]).view(T, nkv, hd), P, 1e6).reshape(T, -1).numpy()
    torch.cuda.synchronize()
    got = to_np(d)
    assert rel_err(got[:, :nh * hd], q) <= TOL
    assert rel_err(got[:, nh * hd:(nh + nkv) * hd], kk) <= TOL
    np.testing.assert_array_equal(got[:, (nh + nkv) * hd:], qkv[:, (nh + nkv) * hd:])
    # backward = transpose of the rotation (pure fp64 autograd)
    g = synth.gaussian_f32((T, ncols), 13, hd)
    out = torch.empty((T, ncols), dtype=torch.bfloat16, device=DEV)
    k("lsk_rope_bwd_cast", torch.from_numpy(g).to(DEV), out, ncols, posd, ct, st, T, nh + nkv, hd, ncols)
    with om.pure_fp64():
        X = om.t64(qkv[:, :(nh + nkv) * hd]).requires_grad_(True)
        y = om.rope(X.view(T, nh + nkv, hd), P, 1e6).reshape(T, -1)
        (y * om.t64(g[:, :(nh + nkv) * hd])).sum().backward()
    torch.cuda.synchronize()
    got = to_np(out)
    assert rel_err(got[:, :(nh + nkv) * hd], X.grad.numpy()) <= TOL
    np.testing.assert_array_equal(got[:, (nh + nkv) * hd:], synth.to_bf16_values(g[:, (nh + nkv) * hd:]))


@pytest.mark.parametrize("T,I", [(3, 64), (512, 4864), (1024, 14336)])
def test_swiglu_fwd_bwd(T, I):
    gu = synth.gaussian((T, 2 * I), 14, I, std=2.0)
    dh = synth.gaussian_f32((T, I), 15, I)
    gd = bf16_dev(gu)
    h = torch.empty((T, I), dtype=torch.bfloat16, device=DEV)
    k("lsk_swiglu_fwd", gd, h, T, I)
    G = om.t64(gu[:, :I]).requires_grad_(True)
    U = om.t64(gu[:, I:]).requires_grad_(True)
    ho = om.swiglu(G, U)
    (ho * om.t64(dh)).sum().backward()
    dgu = torch.empty((T, 2 * I), dtype=torch.bfloat16, device=DEV)
    k("lsk_swiglu_bwd", torch.from_numpy(dh).to(DEV), gd, dgu, T, I)
    torch.cuda.synchronize()
    assert rel_err(to_np(h), ho.detach().numpy()) <= TOL
    got = to_np(dgu)
    assert rel_err(got[:, :I], G.grad.numpy()) <= TOL
    assert rel_err(got[:, I:], U.grad.numpy()) <= TOL


# ------------------------------------------------------------------ attention

ATT_CASES = [
    (64, 14, 2, [0, 512]),
    (128, 32, 8, [0, 512, 1024]),
    (128, 4, 1, [0, 1, 66, 200]),     # length-1 sequence, ragged tiles
    (64, 4, 4, [0, 130]),
    (128, 40, 8, [0, 1000, 2048]),    # 32B head layout, the longest sequence, ragged 128-row tiles
    (64, 16, 2, [0, 0, 300, 1000]),   # an empty sequence among ragged ones
]


@pytest.mark.parametrize("hd,nh,nkv,cu", ATT_CASES)
def test_attention_fwd_bwd(hd, nh, nkv, cu):
    T = cu[-1]
    maxlen = max(b - a for a, b in zip(cu[:-1], cu[1:]))
    ncols = (nh + 2 * nkv) * hd
    qkv = synth.gaussian((T, ncols), 16, hd, nh)
    do = synth.gaussian((T, nh * hd), 17, hd, nh)
    qd = bf16_dev(qkv)
    cud = torch.tensor(cu, dtype=torch.int32, device=DEV)
    o = torch.empty((T, nh * hd), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((nh, T), dtype=torch.float32, device=DEV)
    k("lsk_attn_fwd", qd, ncols, cud, len(cu) - 1, maxlen, nh, nkv, hd, o, nh * hd, lse, T)
    Q = om.t64(qkv[:, :nh * hd]).view(T, nh, hd).requires_grad_(True)
    K_ = om.t64(qkv[:, nh * hd:(nh + nkv) * hd]).view(T, nkv, hd).requires_grad_(True)
    V = om.t64(qkv[:, (nh + nkv) * hd:]).view(T, nkv, hd).requires_grad_(True)
    with om.pure_fp64():
        ref = om.attention(Q, K_, V, cu)
    (ref * om.t64(do).view(T, nh, hd)).sum().backward()
    dscr = torch.empty((nh, T), dtype=torch.float32, device=DEV)
    dq = torch.zeros((T, ncols), dtype=torch.float32, device=DEV)
    dod = bf16_dev(do)
    k("lsk_attn_bwd", qd, ncols, dod, o, nh * hd, lse, cud, len(cu) - 1, maxlen, nh, nkv, hd, dscr, dq, ncols, T,
      None)
    grads = [dq]
    if nh > nkv:
        # dk / dv per query head in separate CTAs, summed in head order by a second kernel
        part = torch.empty((nh // nkv) * T * 2 * nkv * hd, dtype=torch.float32, device=DEV)
        dq2 = torch.zeros((T, ncols), dtype=torch.float32, device=DEV)
        k("lsk_attn_bwd", qd, ncols, dod, o, nh * hd, lse, cud, len(cu) - 1, maxlen, nh, nkv, hd, dscr, dq2, ncols,
          T, part)
        grads.append(dq2)
    torch.cuda.synchronize()
    assert rel_err(to_np(o), ref.detach().reshape(T, -1).numpy()) <= TOL
    for gd in grads:
        g = to_np(gd)
        assert rel_err(g[:, :nh * hd], Q.grad.reshape(T, -1).numpy()) <= TOL
        assert rel_err(g[:, nh * hd:(nh + nkv) * hd], K_.grad.reshape(T, -1).numpy()) <= TOL
        assert rel_err(g[:, (nh + nkv) * hd:], V.grad.reshape(T, -1).numpy()) <= TOL
    if len(grads) == 2:
        # dq is the same kernel either way; dk / dv differ only in summation order
        a_, b_ = to_np(grads[0]), to_np(grads[1])
        assert np.array_equal(a_[:, :nh * hd], b_[:, :nh * hd])
        assert rel_err(b_[:, nh * hd:], a_[:, nh * hd:]) <= 1e-5
    # log-sum-exp of the scaled scores
    lo = to_np(lse)
    for si in range(len(cu) - 1):
        a, b = cu[si], cu[si + 1]
        if b == a:
            continue
        qs = om.t64(qkv[a:b, :nh * hd]).view(b - a, nh, hd).transpose(0, 1)
        ks = om.t64(qkv[a:b, nh * hd:(nh + nkv) * hd]).view(b - a, nkv, hd).transpose(0, 1).repeat_interleave(nh // nkv, 0)
        sc = qs @ ks.transpose(1, 2) / math.sqrt(hd)
        sc = sc.masked_fill(torch.triu(torch.ones(b - a, b - a, dtype=torch.bool), 1), float("-inf"))
        want = torch.logsumexp(sc, -1).numpy()
        assert np.abs(lo[:, a:b] - want).max() <= 1e-3


def test_attention_masks_and_head_groups_exactly():
    """With q = 0 every score is exactly 0, so each row averages the values of exactly the
    keys it may see (causal, inside its own sequence) with weight 1 / (r + 1), and
    lse = ln(r + 1).  The log-sum-exp pins how many keys each row saw to fp32 precision;
    value columns holding the bits of the key's position pin which keys they were; a
    value column holding the key/value head index pins the query-head grouping (exact).
    Ragged sequences, a length-1 one and a 512-long one (four 128-row query tiles)."""
    hd, nh, nkv = 128, 8, 2
    cu = [0, 1, 66, 200, 712]
    T = cu[-1]
    ncols = (nh + 2 * nkv) * hd
    pos = np.concatenate([np.arange(b - a) for a, b in zip(cu[:-1], cu[1:])])
    qkv = np.zeros((T, ncols), np.float32)
    qkv[:, nh * hd:(nh + nkv) * hd] = synth.gaussian((T, nkv * hd), 60, T)   # any keys: q = 0
    for g in range(nkv):
        vc = (nh + nkv + g) * hd
        for b in range(9):
            qkv[:, vc + b] = (pos >> b) & 1
        qkv[:, vc + hd - 1] = g
    qd = bf16_dev(qkv)
    cud = torch.tensor(cu, dtype=torch.int32, device=DEV)
    o = torch.empty((T, nh * hd), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((nh, T), dtype=torch.float32, device=DEV)
    k("lsk_attn_fwd", qd, ncols, cud, len(cu) - 1, 512, nh, nkv, hd, o, nh * hd, lse, T)
    torch.cuda.synchronize()
    got = to_np(o).reshape(T, nh, hd)
    lo = to_np(lse)
    np.testing.assert_allclose(lo, np.broadcast_to(np.log(pos + 1.0), (nh, T)), rtol=0, atol=2e-5)
    for b in range(9):
        # fraction of positions 0..r with bit b set
        bits = (pos >> b) & 1
        want = np.empty(T)
        for a, e in zip(cu[:-1], cu[1:]):
            want[a:e] = np.cumsum(bits[a:e]) / (pos[a:e] + 1.0)
        for h in range(nh):
            assert np.abs(got[:, h, b] - want).max() <= 2.0 ** -8 * np.abs(want).max() + 1e-6, (b, h)
    for h in range(nh):
        assert (got[:, h, hd - 1] == h // (nh // nkv)).all()


# ------------------------------------------------------------------ vocabulary logprobs

@pytest.mark.parametrize("T,H,V", [(64, 256, 512), (300, 896, 3072), (1024, 4096, 128256)])
def test_vocab_logprob_fwd_bwd(T, H, V):
    h = synth.gaussian((T, H), 18, H)
    w = _w(V, H, seed=19)
    p, a, _, _ = nf4_dev(w)
    tgt = np.random.default_rng(20).integers(0, V, T).astype(np.int32)
    tgt[-1] = -1
    tgt[5] = V - 1
    hd_, td = bf16_dev(h), torch.from_numpy(tgt).to(DEV)
    P = (V + 127) // 128
    scr = torch.empty(2 * T * P, dtype=torch.float32, device=DEV)
    tl, lse, lp = (torch.empty(T, dtype=torch.float32, device=DEV) for _ in range(3))
    k("lsk_vocab_logprob", hd_, T, H, p, a, V, td, scr, tl, lse, lp)
    rows = np.arange(T) if T <= 300 else np.array([0, 1, 5, 500, 1022, 1023])
    wd = _oracle_deq(w)
    logits = om.t64(h[rows]) @ om.t64(wd).T
    lse_o = torch.logsumexp(logits, -1).numpy()
    tg = tgt[rows]
    lp_o = np.where(tg >= 0, logits.numpy()[np.arange(len(rows)), np.maximum(tg, 0)] - lse_o, 0.0)
    torch.cuda.synchronize()
    assert np.abs(to_np(lse)[rows] - lse_o).max() <= 2e-2
    assert np.abs(to_np(lp)[rows] - lp_o).max() <= 2e-2
    if T > 300:
        return
    # backward: dh = sum_v coef (onehot - softmax) W
    coef = synth.gaussian_f32((T,), 21, T)
    dl = torch.empty((T, V), dtype=torch.bfloat16, device=DEV)
    dh = torch.empty((T, H), dtype=torch.float32, device=DEV)
    half = (V // 2) // 256 * 256 or V
    k("lsk_vocab_bwd", hd_, T, H, p, a, 0, half, td, lse, torch.from_numpy(coef).to(DEV), dl, dh, 0)
    if half < V:
        off = half * (H // 2)
        k("lsk_vocab_bwd", hd_, T, H, p[off:] if p.dim() == 1 else p.view(-1)[off:],
          a.view(-1)[half * (H // 64):], half, V - half, td, lse, torch.from_numpy(coef).to(DEV), dl, dh, 1)
    sm = torch.softmax(logits, -1).numpy()
    oh = np.zeros_like(sm)
    oh[np.arange(T)[tgt >= 0], tgt[tgt >= 0]] = 1.0
    want = (coef[:, None] * (oh - sm)) @ wd.astype(np.float64)
    torch.cuda.synchronize()
    assert rel_err(to_np(dh), want) <= TOL
