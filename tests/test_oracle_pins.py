"""Pins of the oracle against things other than itself (no GPU needed).

Each test fixes one part of the oracle by a closed form, an invariant, brute
force on a tiny input, a finite difference, or a library special case, so that
a dropped term, a wrong sign or index, or a transposed operand fails here.
"""
import math

import numpy as np
import pytest
import torch
from scipy.stats import norm

import oracle
import synth
from oracle import model as M

F64 = torch.float64


# ------------------------------------------------------------------ NF4 table and rounding

def test_nf4_table_from_normal_quantile_construction():
    """QLoRA Sec. 3: quantiles of N(0,1), 8 positive and 7 negative halves, exact zero,
    normalised to [-1, 1].  The published table must follow from that construction."""
    d = 0.5 * (1 - 1 / (2 * 15)) + 0.5 * (1 - 1 / (2 * 16))
    pos = norm.ppf(np.linspace(d, 0.5, 9)[:-1])
    neg = -norm.ppf(np.linspace(d, 0.5, 8)[:-1])
    v = np.sort(np.concatenate([pos, [0.0], neg]))
    v /= np.abs(v).max()
    np.testing.assert_allclose(oracle.NF4_TABLE, v, rtol=0, atol=1e-6)


def test_nf4_table_structure():
    t = oracle.NF4_TABLE
    assert t.dtype == np.float32 and t.shape == (16,)
    assert np.all(np.diff(t) > 0)
    assert t[0] == -1.0 and t[15] == 1.0 and t[7] == 0.0
    assert (t < 0).sum() == 7 and (t > 0).sum() == 8


def test_bf16_round_matches_library_and_ties():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-30, 30, 100000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(oracle.bf16_round_f32(x), ref)
    # hand cases: 1 + 2^-8 is a tie -> even (1.0); 1 + 3*2^-8 is a tie -> even (1 + 2^-6)
    cases = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 1 + 2.0 ** -8 + 2.0 ** -20],
                     np.float32)
    want = np.array([1.0, 1 + 2.0 ** -6, -1.0, 1 + 2.0 ** -7], np.float32)
    np.testing.assert_array_equal(oracle.bf16_round_f32(cases), want)


# ------------------------------------------------------------------ quantiser

def _brute_codes(w):
    """Pure-Python nearest-code search, one element at a time."""
    n, k = w.shape
    t = [np.float32(v) for v in oracle.NF4_TABLE]
    codes = np.zeros((n, k), np.uint8)
    absmax = np.zeros((n, k // 64), np.float32)
    for i in range(n):
        for b in range(k // 64):
            blk = w[i, b * 64:(b + 1) * 64]
            a = np.float32(max(abs(float(v)) for v in blk))
            absmax[i, b] = a
            for j, v in enumerate(blk):
                if a == 0:
                    codes[i, b * 64 + j] = 7
                    continue
                x = np.float32(v / a)
                best, bi = None, 0
                for ci, q in enumerate(t):
                    dd = np.float32(abs(np.float32(x - q)))
                    if best is None or dd < best:
                        best, bi = dd, ci
                codes[i, b * 64 + j] = bi
    return codes, absmax


def test_quantize_brute_force():
    rng = np.random.default_rng(2)
    w = (rng.standard_normal((3, 192)) * 0.02).astype(np.float32)
    w[1, 64:128] = 0.0                     # an all-zero block
    w[2, :8] = [0.5, -0.5, 0.25, 0, 1e-30, -1e-30, 0.5, -0.5]
    c, a = oracle.nf4_quantize(w)
    cb, ab = _brute_codes(w)
    np.testing.assert_array_equal(a, ab)
    np.testing.assert_array_equal(c, cb)


def test_quantize_edge_cases():
    t = oracle.NF4_TABLE
    w = np.zeros((4, 64), np.float32)
    w[0, :16] = t * np.float32(2.0)          # exact table values times absmax 2
    w[1, 0], w[1, 1] = 3.0, -3.0             # +/- absmax -> codes 15 and 0
    mids = ((t[:-1].astype(np.float64) + t[1:]) / 2).astype(np.float32)
    w[2, :15] = mids                          # midpoints (absmax 1 set below) -> lower index
    w[2, 15] = 1.0
    # row 3 stays all zero -> code 7, absmax 0
    c, a = oracle.nf4_quantize(w)
    np.testing.assert_array_equal(c[0, :16], np.arange(16))
    assert c[1, 0] == 15 and c[1, 1] == 0
    x = (mids / np.float32(1.0)).astype(np.float32)
    d_lo = np.abs(x - t[:-1]).astype(np.float32)
    d_hi = np.abs(x - t[1:]).astype(np.float32)
    want = np.where(d_hi < d_lo, np.arange(1, 16), np.arange(15))
    np.testing.assert_array_equal(c[2, :15], want)
    assert np.all(c[3] == 7) and a[3, 0] == 0.0
    np.testing.assert_array_equal(oracle.nf4_dequantize(c, a)[3], np.zeros(64, np.float32))


def test_pack_nibble_order_and_roundtrip():
    codes = np.array([[1, 2, 15, 0]], np.uint8)
    p = oracle.nf4_pack(codes)
    assert p.tolist() == [[0x12, 0xF0]]
    rng = np.random.default_rng(3)
    c = rng.integers(0, 16, (5, 128), dtype=np.uint8)
    np.testing.assert_array_equal(oracle.nf4_unpack(oracle.nf4_pack(c)), c)


def test_dequant_closed_form():
    t = oracle.NF4_TABLE
    codes = np.tile(np.arange(16, dtype=np.uint8), 4)[None, :]
    absmax = np.array([[0.5]], np.float32)
    d = oracle.nf4_dequantize(codes, absmax)
    assert d[0, 15] == 0.5 and d[0, 0] == -0.5 and d[0, 7] == 0.0
    # one fp32 multiply then one bf16 rounding (round half to even)
    a = np.float32(0.0123456)
    want = torch.tensor(np.float32(t[13]) * a).to(torch.bfloat16).float().item()
    assert oracle.nf4_dequantize(np.full((1, 64), 13, np.uint8), np.array([[a]]))[0, 0] == want
    # quantisation error bound: |w - deq| <= absmax * (max gap / 2) + bf16 rounding
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((8, 256)) * 0.02).astype(np.float32)
    c, a = oracle.nf4_quantize(w)
    err = np.abs(oracle.nf4_dequantize(c, a) - w).reshape(8, 4, 64).max(axis=2)
    gap = np.diff(t).max() / 2
    assert np.all(err <= a * gap * 1.01 + a * 2.0 ** -8)


# ------------------------------------------------------------------ blocks

def test_rmsnorm_hand_value_and_scale_invariance():
    x = torch.tensor([[3.0, 4.0]], dtype=F64)
    w = torch.tensor([1.0, 2.0], dtype=F64)
    with M.pure_fp64():
        y = M.rmsnorm(x, w, 0.0)
    r = 1 / math.sqrt(12.5)
    np.testing.assert_allclose(y.numpy(), [[3 * r, 8 * r]], rtol=1e-15)
    rng = np.random.default_rng(5)
    x = torch.from_numpy(rng.standard_normal((4, 64)))
    w = torch.from_numpy(rng.standard_normal(64))
    np.testing.assert_array_equal(M.rmsnorm(x * 8.0, w, 0.0).numpy(), M.rmsnorm(x, w, 0.0).numpy())


def test_rope_identity_norm_and_relative_position():
    rng = np.random.default_rng(6)
    x = M.bf16r(torch.from_numpy(rng.standard_normal((6, 2, 8))))
    y = M.rope(x, torch.zeros(6, dtype=torch.long), 1e4)
    np.testing.assert_array_equal(y.numpy(), x.numpy())           # position 0 = identity
    with M.pure_fp64():
        pos = torch.arange(6)
        y = M.rope(x, pos, 1e4)
        # pairs (i, i + hd/2) are rotated: per-pair norm preserved
        n0 = x[..., :4] ** 2 + x[..., 4:] ** 2
        n1 = y[..., :4] ** 2 + y[..., 4:] ** 2
        np.testing.assert_allclose(n1.numpy(), n0.numpy(), rtol=1e-12)
        # hd = 2, theta^0 = 1: a plain rotation by angle = position
        z = torch.tensor([[[1.0, 0.0]]], dtype=F64).repeat(3, 1, 1)
        r = M.rope(z, torch.tensor([0, 1, 2]), 10.0)
        np.testing.assert_allclose(r[:, 0, 0].numpy(), np.cos([0, 1, 2]), rtol=1e-14)
        np.testing.assert_allclose(r[:, 0, 1].numpy(), np.sin([0, 1, 2]), atol=1e-15)
        # <rope(q, m), rope(k, n)> depends on m - n only
        q = torch.from_numpy(rng.standard_normal((1, 1, 8)))
        k = torch.from_numpy(rng.standard_normal((1, 1, 8)))
        def dot(m, n):
            return float((M.rope(q, torch.tensor([m]), 1e4) * M.rope(k, torch.tensor([n]), 1e4)).sum())
        assert abs(dot(5, 2) - dot(13, 10)) < 1e-12
        assert abs(dot(5, 2) - dot(2, 5)) > 1e-6


def _attention_brute(q, k, v, cu):
    T, nh, hd = q.shape
    kv = k.shape[1]
    out = np.zeros((T, nh, hd))
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        for h in range(nh):
            g = h * kv // nh
            for t in range(a, b):
                sc = [float(np.dot(q[t, h], k[j, g])) / math.sqrt(hd) for j in range(a, t + 1)]
                m = max(sc)
                e = [math.exp(x - m) for x in sc]
                z = sum(e)
                for jj, j in enumerate(range(a, t + 1)):
                    out[t, h] += e[jj] / z * v[j, g]
    return out


def test_attention_brute_force_gqa_varlen():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((7, 4, 8))
    k = rng.standard_normal((7, 2, 8))
    v = rng.standard_normal((7, 2, 8))
    cu = [0, 3, 7]
    with M.pure_fp64():
        o = M.attention(torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), cu)
    np.testing.assert_allclose(o.numpy(), _attention_brute(q, k, v, cu), rtol=1e-12, atol=1e-13)
    # first position of each sequence attends only to itself: o = v
    for a in cu[:-1]:
        np.testing.assert_allclose(o[a].numpy(), np.repeat(v[a], 2, axis=0), rtol=1e-14)


def test_swiglu_closed_form():
    g = torch.tensor([0.0, 1.0, -2.0, 30.0], dtype=F64)
    u = torch.tensor([5.0, 2.0, 1.0, 1.0], dtype=F64)
    with M.pure_fp64():
        h = M.swiglu(g, u).numpy()
    want = [0.0, 2.0 / (1 + math.exp(-1)), -2.0 / (1 + math.exp(2)), 30.0 / (1 + math.exp(-30))]
    np.testing.assert_allclose(h, want, rtol=1e-15)


def test_lora_linear_closed_forms():
    """B = 0 gives the base output exactly; gradients match their closed forms."""
    rng = np.random.default_rng(8)
    x = synth.gaussian((16, 128), 0, 1)
    w = oracle.nf4_dequantize(*oracle.nf4_quantize((rng.standard_normal((96, 128)) * 0.02).astype(np.float32)))
    a = synth.gaussian((4, 128), 0, 2, std=0.01)
    b = synth.gaussian((96, 4), 0, 3, std=0.01)
    dy = synth.gaussian((16, 96), 0, 4)
    s = 2.0
    base = M.linear(M.t64(x), M.t64(w)).numpy()
    r0 = M.lora_linear_step(x, w, a, np.zeros_like(b), s, dy)
    np.testing.assert_array_equal(r0["y"].numpy(), base)
    with M.pure_fp64():
        r = M.lora_linear_step(x, w, a, b, s, dy)
    X, W, A, B, DY = (x.astype(np.float64), w.astype(np.float64), a.astype(np.float64),
                      b.astype(np.float64), dy.astype(np.float64))
    u = s * X @ A.T
    np.testing.assert_allclose(r["y"].numpy(), X @ W.T + u @ B.T, rtol=1e-12)
    np.testing.assert_allclose(r["db"].numpy(), DY.T @ u, rtol=1e-12)
    du = DY @ B
    np.testing.assert_allclose(r["da"].numpy(), s * du.T @ X, rtol=1e-12)
    np.testing.assert_allclose(r["dx"].numpy(), DY @ W + s * du @ A, rtol=1e-12)


# ------------------------------------------------------------------ stack, losses, gradients

TINY = synth.StackConfig("tiny", layers=2, hidden=64, heads=4, kv_heads=2, head_dim=16, inter=128,
                         vocab=40, tied=True, rope_theta=1e4, eps=1e-6, lora_r=2, lora_alpha=4.0,
                         seq_len=6, nseq=2, prompt_len=2, method="dpo", beta=0.5)


def _tiny(cfg=TINY, zero_b=False, seed=0):
    sw = M.build_stack(cfg, seed, synth)
    ads = M.build_adapters(cfg, seed, synth, zero_b=zero_b)
    # larger adapters so the finite differences see a clear signal
    for ad in ads:
        for p in ad.params():
            p.data.mul_(30.0)
    return sw, ads


def test_logprobs_normalise_and_adapter_off_equals_base():
    cfg = TINY
    sw, ads = _tiny()
    tok = synth.tokens(cfg)
    cu = synth.seq_offsets(cfg)
    tr = {}
    off = M.stack_forward(tok, cu, sw, ads, cfg, adapter_on=False, trace=tr)
    p = torch.exp(tr["logits"] - off["lse"][:, None]).sum(dim=1)
    np.testing.assert_allclose(p.numpy(), 1.0, rtol=1e-13)
    base = M.stack_forward(tok, cu, sw, None, cfg)
    np.testing.assert_array_equal(off["lp"].numpy(), base["lp"].numpy())
    _, zb = _tiny(zero_b=True)
    on0 = M.stack_forward(tok, cu, sw, zb, cfg, adapter_on=True)
    np.testing.assert_array_equal(on0["lp"].numpy(), base["lp"].numpy())
    on = M.stack_forward(tok, cu, sw, ads, cfg, adapter_on=True)
    assert not np.array_equal(on["lp"].numpy(), base["lp"].numpy())


def test_sft_loss_uniform_logits_is_log_vocab():
    cfg = TINY.with_(method="sft", prompt_len=0)
    sw, ads = _tiny(cfg)
    sw.lm_head = torch.zeros_like(sw.lm_head)
    tok = synth.tokens(cfg)
    r = M.stack_forward(tok, synth.seq_offsets(cfg), sw, ads, cfg)
    loss = M.sft_loss(r["lp"], synth.loss_mask(cfg))
    assert abs(float(loss) - math.log(cfg.vocab)) < 1e-14


def test_dpo_ln2_at_policy_equals_reference_and_gradient_sign():
    cfg = TINY
    sw, zb = _tiny(zero_b=True)
    out = M.train_step(synth.tokens(cfg), synth.seq_offsets(cfg), synth.loss_mask(cfg), sw, zb, cfg)
    assert float(out["loss"]) == pytest.approx(math.log(2.0), abs=1e-15)
    pi = torch.tensor([0.0, 0.0], dtype=F64, requires_grad=True)
    ref = torch.tensor([0.0, 0.0], dtype=F64)
    L = M.dpo_loss(pi, ref, 0.1)
    L.backward()
    # dL/dpi_c = -beta sigma(-z) < 0, dL/dpi_r = +beta sigma(-z) > 0; at z = 0, sigma = 1/2
    np.testing.assert_allclose(pi.grad.numpy(), [-0.05, 0.05], rtol=1e-15)
    big = M.dpo_loss(torch.tensor([1e4, -1e4], dtype=F64), ref, 1.0)
    assert torch.isfinite(big) and float(big) < 1e-300 + 1e-12
    neg = M.dpo_loss(torch.tensor([-1e4, 1e4], dtype=F64), ref, 1.0)
    assert float(neg) == pytest.approx(2e4, rel=1e-12)


@pytest.mark.parametrize("method", ["sft", "dpo"])
def test_lora_grads_finite_differences(method):
    cfg = TINY.with_(method=method, prompt_len=2 if method == "dpo" else 0)
    sw, ads = _tiny(cfg)
    tok, cu, mask = synth.tokens(cfg), synth.seq_offsets(cfg), synth.loss_mask(cfg)
    with M.pure_fp64():
        out = M.train_step(tok, cu, mask, sw, ads, cfg)

        def loss_at():
            with torch.no_grad():
                pol = M.stack_forward(tok, cu, sw, ads, cfg, True)
                if method == "sft":
                    return float(M.sft_loss(pol["lp"], mask))
                ref = M.stack_forward(tok, cu, sw, ads, cfg, False)
                return float(M.dpo_loss(M.seq_sums(pol["lp"], mask, cu),
                                        M.seq_sums(ref["lp"], mask, cu), cfg.beta))

        rng = np.random.default_rng(9)
        h = 1e-6
        for li in range(cfg.layers):
            for pi, p in enumerate(ads[li].params()):
                g = out["grads"][li][pi]
                for _ in range(3):
                    idx = tuple(int(rng.integers(0, s)) for s in p.shape)
                    old = p.data[idx].item()
                    p.data[idx] = old + h
                    lp_ = loss_at()
                    p.data[idx] = old - h
                    lm_ = loss_at()
                    p.data[idx] = old
                    fd = (lp_ - lm_) / (2 * h)
                    scale = float(g.abs().max()) + 1e-12
                    assert abs(fd - float(g[idx])) <= 1e-6 * scale + 1e-9, (li, pi, idx, fd, float(g[idx]))


def _rope_complex(x, pos, theta):
    """RoPE as complex multiplication: (x_i + j x_{i+hd/2}) * exp(j pos theta^(-2i/hd))."""
    hd = x.shape[-1]
    half = hd // 2
    z = torch.complex(x[..., :half], x[..., half:])
    ang = pos.to(F64)[:, None] * theta ** (-torch.arange(0, hd, 2, dtype=F64) / hd)[None, :]
    z = z * torch.polar(torch.ones_like(ang), ang)[:, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


def test_decoder_layer_matches_library_composition():
    """The layer wiring against torch's rms_norm / scaled_dot_product_attention / silu."""
    import torch.nn.functional as F
    cfg = TINY
    sw, ads = _tiny()
    lw, ad = sw.layers[0], ads[0]
    cu = [0, 5, 12]
    T = cu[-1]
    x = M.t64(synth.gaussian((T, cfg.hidden), 0, 11))
    s = cfg.lora_scale
    with M.pure_fp64():
        got = M.decoder_layer(x, lw, ad, cfg, cu, adapter_on=True)
    H, nh, kv, hd = cfg.hidden, cfg.heads, cfg.kv_heads, cfg.head_dim
    n1 = F.rms_norm(x, (H,), lw.w1, cfg.eps)
    q = F.linear(n1, lw.wq) + s * F.linear(F.linear(n1, ad.aq), ad.bq)
    k = F.linear(n1, lw.wk)
    v = F.linear(n1, lw.wv) + s * F.linear(F.linear(n1, ad.av), ad.bv)
    pos = torch.cat([torch.arange(cu[i + 1] - cu[i]) for i in range(len(cu) - 1)])
    q = _rope_complex(q.view(T, nh, hd), pos, cfg.rope_theta)
    k = _rope_complex(k.view(T, kv, hd), pos, cfg.rope_theta)
    v = v.view(T, kv, hd)
    o = torch.cat([F.scaled_dot_product_attention(
        q[a:b].transpose(0, 1)[None], k[a:b].transpose(0, 1)[None], v[a:b].transpose(0, 1)[None],
        is_causal=True, enable_gqa=True)[0].transpose(0, 1) for a, b in zip(cu[:-1], cu[1:])])
    x1 = x + F.linear(o.reshape(T, nh * hd), lw.wo)
    n2 = F.rms_norm(x1, (H,), lw.w2, cfg.eps)
    want = x1 + F.linear(F.silu(F.linear(n2, lw.wg)) * F.linear(n2, lw.wu), lw.wd)
    np.testing.assert_allclose(got.detach().numpy(), want.detach().numpy(), rtol=1e-11, atol=1e-12)


def test_logprobs_match_cross_entropy_and_dpo_matches_logsigmoid():
    import torch.nn.functional as F
    cfg = TINY
    sw, ads = _tiny()
    tok, cu = synth.tokens(cfg), synth.seq_offsets(cfg)
    tr = {}
    r = M.stack_forward(tok, cu, sw, ads, cfg, trace=tr)
    y = M.targets(tok, cu)
    has = y >= 0
    ce = F.cross_entropy(tr["logits"][torch.from_numpy(has)], torch.from_numpy(y[has]), reduction="none")
    np.testing.assert_allclose(-r["lp"][torch.from_numpy(has)].detach().numpy(), ce.detach().numpy(), rtol=1e-13)
    assert np.all(r["lp"][torch.from_numpy(~has)].detach().numpy() == 0)
    pi = torch.tensor([-3.0, -5.0, -2.0, -2.5], dtype=F64)
    ref = torch.tensor([-4.0, -4.5, -2.2, -2.0], dtype=F64)
    z = 0.3 * ((pi[0::2] - ref[0::2]) - (pi[1::2] - ref[1::2]))
    np.testing.assert_allclose(float(M.dpo_loss(pi, ref, 0.3)), float(-F.logsigmoid(z).mean()), rtol=1e-15)


def test_causality_and_sequence_independence():
    cfg = TINY
    sw, ads = _tiny()
    tok, cu = synth.tokens(cfg), synth.seq_offsets(cfg)
    base = M.stack_forward(tok, cu, sw, ads, cfg)["lp"].detach().numpy()
    # changing token 4 of sequence 0 leaves predictions at positions 0..2 unchanged
    t2 = tok.copy()
    t2[4] = (t2[4] + 1) % cfg.vocab
    ch = M.stack_forward(t2, cu, sw, ads, cfg)["lp"].detach().numpy()
    np.testing.assert_array_equal(ch[:3], base[:3])
    assert not np.array_equal(ch[3:6], base[3:6])
    np.testing.assert_array_equal(ch[6:], base[6:])           # other sequence untouched
    # sequence 1 run alone gives the same logprobs as inside the two-sequence pass
    alone = M.stack_forward(tok[6:], [0, 6], sw, ads, cfg)["lp"].detach().numpy()
    np.testing.assert_array_equal(alone, base[6:])


def test_accumulate_in_fp32_computes_the_same_step():
    """The fp32-accumulation mode (used to measure rounding floors) is the same
    computation: on a tiny stack without bf16 storage it matches fp64 to fp32 accuracy,
    and the context restores fp64 afterwards."""
    cfg = TINY.with_(method="dpo", prompt_len=2)
    sw, ads = _tiny(cfg)
    tok, cu, mask = synth.tokens(cfg), synth.seq_offsets(cfg), synth.loss_mask(cfg)
    with M.pure_fp64():
        o64 = M.train_step(tok, cu, mask, sw, ads, cfg)
        with M.accumulate_in(torch.float32):
            o32 = M.train_step(tok, cu, mask, M.cast_stack(sw, torch.float32),
                               M.cast_adapters(ads, torch.float32), cfg)
            assert o32["lp"].dtype == torch.float32
    assert M.t64(np.zeros(2)).dtype == F64
    assert float(o32["loss"]) == pytest.approx(float(o64["loss"]), rel=1e-5)
    g64 = torch.cat([g.ravel() for l in o64["grads"] for g in l])
    g32 = torch.cat([g.ravel().double() for l in o32["grads"] for g in l])
    assert float((g32 - g64).abs().max() / g64.abs().max()) < 1e-4


# ------------------------------------------------------------------ golden fixtures

GOLDEN = __import__("os").path.join(__import__("os").path.dirname(__file__), "golden")


def test_nf4_table_matches_published_fixture():
    vals = [float(l) for l in open(f"{GOLDEN}/nf4_table.txt") if l.strip() and not l.startswith("#")]
    np.testing.assert_array_equal(oracle.NF4_TABLE, np.array(vals, np.float32))


def test_oracle_reproduces_tiny_dpo_golden():
    import json
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", f"{GOLDEN}/make_golden.py")
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    want = json.load(open(f"{GOLDEN}/tiny_dpo_step.json"))
    got = mg.tiny_dpo_step()
    assert got["config"] == want["config"]
    assert got["loss"] == pytest.approx(want["loss"], rel=1e-12)
    np.testing.assert_allclose(got["pi"], want["pi"], rtol=1e-12)
    np.testing.assert_allclose(got["ref"], want["ref"], rtol=1e-12)
    np.testing.assert_allclose(got["grad_norms"], want["grad_norms"], rtol=1e-10)
    np.testing.assert_allclose(got["grad_head"], want["grad_head"], rtol=1e-9, atol=1e-15)


# ------------------------------------------------------------------ SimPO, ORPO, KTO

def test_simpo_closed_forms():
    counts = torch.tensor([4.0, 8.0], dtype=F64)
    # equal average logprobs and no margin: -log sigmoid(0) = ln 2
    pi = torch.tensor([-8.0, -16.0], dtype=F64, requires_grad=True)
    L = M.simpo_loss(pi, counts, beta=2.0, gamma=0.0)
    assert float(L.detach()) == pytest.approx(math.log(2.0), rel=1e-15)
    L.backward()
    # dL/dpi_c = -sigma(-z) beta / |c|, dL/dpi_r = +sigma(-z) beta / |r|, sigma(0) = 1/2
    np.testing.assert_allclose(pi.grad.numpy(), [-0.5 * 2.0 / 4, 0.5 * 2.0 / 8], rtol=1e-15)
    # the margin gamma shifts the logit: z = -gamma
    L2 = M.simpo_loss(pi.detach(), counts, beta=2.0, gamma=1.5)
    assert float(L2) == pytest.approx(math.log1p(math.exp(1.5)), rel=1e-14)
    # length normalisation: doubling a sequence's sum and its length changes nothing
    a = M.simpo_loss(torch.tensor([-3.0, -5.0], dtype=F64), torch.tensor([3.0, 5.0], dtype=F64), 1.0, 0.2)
    b = M.simpo_loss(torch.tensor([-6.0, -5.0], dtype=F64), torch.tensor([6.0, 5.0], dtype=F64), 1.0, 0.2)
    assert float(a) == pytest.approx(float(b), rel=1e-15)


def test_orpo_closed_forms():
    counts = torch.tensor([2.0, 2.0], dtype=F64)
    pi = torch.tensor([-1.0, -3.0], dtype=F64)
    # lambda = 0: the chosen response's mean NLL
    assert float(M.orpo_loss(pi, counts, 0.0)) == pytest.approx(0.5, rel=1e-15)
    # log odds against log(P / (1 - P)) computed directly
    lc, lr = -0.5, -1.5
    odds = lambda l: math.log(math.exp(l) / (1 - math.exp(l)))
    want = 0.5 + 0.1 * math.log1p(math.exp(-(odds(lc) - odds(lr))))
    assert float(M.orpo_loss(pi, counts, 0.1)) == pytest.approx(want, rel=1e-13)
    # equal responses: odds-ratio term = ln 2
    eq = M.orpo_loss(torch.tensor([-2.0, -2.0], dtype=F64), counts, 1.0)
    assert float(eq) == pytest.approx(1.0 + math.log(2.0), rel=1e-14)


def test_kto_closed_forms_and_reference_point():
    d = torch.tensor([1, 0], dtype=torch.uint8)
    # policy = reference: r = 0, z0 = 0, sigma(0) = 1/2 -> loss = mean(lambda / 2)
    z = torch.zeros(2, dtype=F64)
    pi = torch.zeros(2, dtype=F64, requires_grad=True)
    L = M.kto_loss(pi, z, d, beta=0.1, lam_d=1.0, lam_u=3.0)
    assert float(L.detach()) == pytest.approx((0.5 + 1.5) / 2, rel=1e-15)
    L.backward()
    # dL/dpi = -lam_d beta s(1-s) / n for desirable, +lam_u beta s(1-s) / n for undesirable
    np.testing.assert_allclose(pi.grad.numpy(), [-1.0 * 0.1 * 0.25 / 2, 3.0 * 0.1 * 0.25 / 2], rtol=1e-15)
    # the reference point is clamped at zero and carries no gradient
    pi2 = torch.tensor([-4.0, -2.0], dtype=F64, requires_grad=True)
    L2 = M.kto_loss(pi2, z, d, beta=1.0, lam_d=1.0, lam_u=1.0)
    want = ((1 - 1 / (1 + math.exp(4.0))) + (1 - 1 / (1 + math.exp(-2.0)))) / 2
    assert float(L2.detach()) == pytest.approx(want, rel=1e-14)
    L2.backward()
    s1 = 1 / (1 + math.exp(4.0))
    s2 = 1 / (1 + math.exp(-2.0))
    np.testing.assert_allclose(pi2.grad.numpy(), [-s1 * (1 - s1) / 2, s2 * (1 - s2) / 2], rtol=1e-13)


@pytest.mark.parametrize("method", ["simpo", "orpo", "kto"])
def test_preference_grads_finite_differences(method):
    cfg = TINY.with_(method=method, prompt_len=2, beta=0.5, simpo_gamma=0.3, orpo_lambda=0.5)
    sw, ads = _tiny(cfg)
    tok, cu, mask = synth.tokens(cfg), synth.seq_offsets(cfg), synth.loss_mask(cfg)
    with M.pure_fp64():
        out = M.train_step(tok, cu, mask, sw, ads, cfg)

        def loss_at():
            with torch.no_grad():
                pi = M.seq_sums(M.stack_forward(tok, cu, sw, ads, cfg, True)["lp"], mask, cu)
                n = M.seq_counts(mask, cu)
                if method == "simpo":
                    return float(M.simpo_loss(pi, n, cfg.beta, cfg.simpo_gamma))
                if method == "orpo":
                    return float(M.orpo_loss(pi, n, cfg.orpo_lambda))
                ref = M.seq_sums(M.stack_forward(tok, cu, sw, ads, cfg, False)["lp"], mask, cu)
                return float(M.kto_loss(pi, ref, M.pair_desirable(len(cu) - 1), cfg.beta, 1.0, 1.0))

        assert float(out["loss"]) == pytest.approx(loss_at(), rel=1e-12)
        rng = np.random.default_rng(11)
        h = 1e-6
        for li in range(cfg.layers):
            for pi_, p in enumerate(ads[li].params()):
                g = out["grads"][li][pi_]
                for _ in range(2):
                    idx = tuple(int(rng.integers(0, s)) for s in p.shape)
                    old = p.data[idx].item()
                    p.data[idx] = old + h
                    lp_ = loss_at()
                    p.data[idx] = old - h
                    lm_ = loss_at()
                    p.data[idx] = old
                    fd = (lp_ - lm_) / (2 * h)
                    scale = float(g.abs().max()) + 1e-12
                    assert abs(fd - float(g[idx])) <= 1e-6 * scale + 1e-9, (li, pi_, idx, fd, float(g[idx]))


def test_adamw_matches_torch_optim():
    """The oracle's AdamW against torch.optim.AdamW (fp64) over three steps."""
    rng = np.random.default_rng(5)
    p0 = torch.from_numpy(rng.normal(size=(7, 5)))
    grads = [torch.from_numpy(rng.normal(size=(7, 5))) for _ in range(3)]
    q = p0.clone().requires_grad_(True)
    opt = torch.optim.AdamW([q], lr=1e-2, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.05)
    p = p0.clone()
    m = torch.zeros_like(p)
    v = torch.zeros_like(p)
    for t, g in enumerate(grads, start=1):
        q.grad = g.clone()
        opt.step()
        M.adamw_update(p, g, m, v, t, 1e-2, 0.9, 0.999, 1e-8, 0.05)
        np.testing.assert_allclose(p.numpy(), q.detach().numpy(), rtol=1e-12, atol=1e-15)
