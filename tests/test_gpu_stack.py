"""Whole-step parity of the streamed CUDA path against the oracle, and the method's
invariants (GPU required).

What the Soup pages fix and these tests check:
  - a streamed pass equals a resident (non-streamed) pass bit for bit (axbrief.com,
    "Beyond Memory: The Layer Streaming Breakthrough"; the evermx.com summary's
    Colab check);
  - the DPO reference logprobs are the frozen base's: the same streamed weights
    with the adapter switched off (Show HN: Fine-tune an 8B model on a 4 GB laptop
    GPU, opening paragraph), so adapter-off = no adapter = B = 0, bit for bit;
  - at policy = reference the DPO loss is ln 2.
Against the oracle (normwise relative error max|gpu - oracle| / max|oracle|), stage
by stage -- the oracle recomputes each decoder layer and the vocabulary head from the
GPU's own stored input of it: every layer's output <= 1e-2, per-token logprobs and
log-sum-exp <= 2e-2 absolute, and the loss from those logprobs <= 1e-2 relative.
The whole step free-running: loss <= 1e-2 relative and LoRA gradients <= 1e-2, or
twice the spread that rounding alone puts on them where that is larger (measured per
case by re-running the oracle with fp32 accumulation: at two 8B-wide layers it moves
the DPO loss by 2.6% and the gradients by 2.0%); free-running logprobs <= 2e-2 on the
shallow stacks, where that floor is below the bound.
"""
import math

import numpy as np
import pytest
import torch

import layer_streamed_nf4_dequant_b300 as L
import synth
from oracle import model as om

from gpu_util import DEV, rel_err, to_np

pytestmark = pytest.mark.gpu

TOL_GRAD = 1e-2
TOL_LP = 2e-2
TOL_LOSS = 1e-2

SMALL_DPO = synth.StackConfig("tiny-dpo", layers=3, hidden=256, heads=4, kv_heads=2, head_dim=64, inter=512,
                              vocab=1024, tied=False, rope_theta=1e4, eps=1e-6, lora_r=16, lora_alpha=32.0,
                              seq_len=96, nseq=4, prompt_len=40, method="dpo", beta=0.1)


def _stack(cfg, resident=False, vocab_chunk_rows=0, zero_b=False, adapters=True, **kw):
    st = L.Stack(cfg, device="cuda:0", resident=resident, vocab_chunk_rows=vocab_chunk_rows, **kw)
    st.load_synthetic(synth, 0)
    if adapters:
        st.set_adapters_synthetic(synth, 0, zero_b=zero_b)
    return st


def _batch(cfg, seed=0, cu=None):
    tok = synth.tokens(cfg, seed)
    if cu is None:
        cu = synth.seq_offsets(cfg)
        mask = synth.loss_mask(cfg)
    else:
        cu = np.asarray(cu, np.int32)
        tok = tok[: cu[-1]]
        mask = np.ones(cu[-1], np.uint8)
        mask[cu[1:] - 1] = 0
    return tok, cu, mask


def _gpu_step(st, cfg, tok, cu, mask):
    t, c, m = st.upload_batch(tok, cu, mask)
    if cfg.method == "dpo":
        o = st.dpo_step(t, c, m, cfg.beta)
    else:
        o = st.sft_step(t, c, m, float(mask.sum()))
    g = st.grads(zero_after=True)
    lp_last, lse_last = st.logprobs(len(tok))
    assert st.sync(300000) == 0, L.last_error(st.ctx)
    return o, g, lp_last, lse_last


def _oracle_step(cfg, tok, cu, mask, zero_b=False):
    sw = om.build_stack(cfg, 0, synth)
    ads = om.build_adapters(cfg, 0, synth, zero_b=zero_b)
    o = om.train_step(tok, cu, mask, sw, ads, cfg)
    flat = np.concatenate([x.numpy().ravel() for layer in o["grads"] for x in layer])
    return o, flat


# ------------------------------------------------------------------ oracle parity

# (config, vocabulary chunk rows, sequence offsets, free-running logprob check)
PARITY = [
    # DPO on a tiny stack, vocabulary split over several streamed chunks
    (SMALL_DPO, 256, None, True),
    # SFT, tied vocabulary, three ragged sequences (T = 300 is not a tile multiple)
    (SMALL_DPO.with_(name="tiny-sft-ragged", method="sft", prompt_len=0, tied=True, nseq=3, seq_len=100),
     512, [0, 100, 237, 300], True),
    # two layers at the full Qwen2.5-3B widths, reduced vocabulary, SFT over 512 tokens
    (synth.small_stack(synth.QWEN_3B, layers=2, vocab=4096, seq_len=512), 0, None, False),
    # two layers at the full Llama-3.1-8B widths, reduced vocabulary, DPO on one pair
    (synth.small_stack(synth.LLAMA_8B, layers=2, vocab=8192, seq_len=512, nseq=2, prompt_len=256), 0, None, False),
    # the single 896-wide decoder layer (14 / 2 heads, SwiGLU 4864) in the tied 151936-row
    # vocabulary of the shape it matches, SFT over 512 tokens
    (synth.LAYER_896, 0, None, True),
]


def _oracle_from_inputs(cfg, tok, cu, sw, ads, xs, adapter_on):
    """Recompute every decoder layer and the vocabulary head in the oracle from the
    GPU's own stored input of each (xs: the L+1 activation-store entries, bf16 values
    as fp64).  Returns the worst normwise layer-output error and the oracle's
    per-token logprobs and log-sum-exp from the GPU's last hidden state."""
    emb = sw.embed[torch.from_numpy(tok.astype(np.int64))]
    worst_layer = rel_err(xs[0].numpy(), emb.numpy())
    with torch.no_grad():
        for l in range(cfg.layers):
            y = om.decoder_layer(xs[l], sw.layers[l], ads[l], cfg, cu, adapter_on)
            worst_layer = max(worst_layer, rel_err(xs[l + 1].numpy(), y.numpy()))
        hf = om.rmsnorm(xs[-1], sw.wf, cfg.eps)
        logits = hf @ sw.lm_head.T
        lse_o = torch.logsumexp(logits, dim=-1)
        y = om.targets(tok, cu)
        lp_o = np.where(y >= 0, logits.numpy()[np.arange(len(tok)), np.maximum(y, 0)] - lse_o.numpy(), 0.0)
    return worst_layer, lp_o, lse_o.numpy()


def _teacher_forced(st, cfg, tok, cu, mask, sw, ads, adapter_on):
    """Run one saved forward on the GPU; recompute every layer and the vocabulary head
    in the oracle from the GPU's own stored input of that layer.  Returns the worst
    normwise layer-output error, the worst per-token logprob / log-sum-exp error, the
    GPU's logprobs and the oracle's teacher-forced logprobs."""
    t, c, m = st.upload_batch(tok, cu, mask)
    st.fwd(t, c, m, adapter_on=adapter_on, save=True)
    lp, lse = st.logprobs(len(tok))
    acts = [st.activation(l, len(tok)) for l in range(cfg.layers + 1)]
    assert st.sync(300000) == 0, L.last_error(st.ctx)
    xs = [om.t64(a.float().cpu().numpy()) for a in acts]
    worst_layer, lp_o, lse_o = _oracle_from_inputs(cfg, tok, cu, sw, ads, xs, adapter_on)
    lp_err = max(np.abs(to_np(lp) - lp_o).max(), np.abs(to_np(lse) - lse_o).max())
    return worst_layer, lp_err, lp, torch.from_numpy(lp_o)


def _teacher_forced_shared(st, cfg, tok, cu, sw, ads, lp2, lse2):
    """The shared-read DPO sweep that produced the step's loss, stage by stage: the
    policy rows' layer inputs are the activation store, the reference rows' come from
    the reference capture (Stack.capture_reference, set before the step); lp2 / lse2
    are that sweep's 2T per-token values.  Returns, per half (True = policy), the worst
    layer error, the worst logprob / LSE error and the oracle's logprobs."""
    T, H = len(tok), cfg.hidden
    pol = [st.activation(l, T) for l in range(cfg.layers + 1)]
    assert st.sync(300000) == 0, L.last_error(st.ctx)
    cap = st.ref_capture[: (cfg.layers + 1) * T * H].view(cfg.layers + 1, T, H)
    out = {}
    for on, acts, rows in ((True, pol, slice(0, T)), (False, list(cap), slice(T, 2 * T))):
        xs = [om.t64(a.float().cpu().numpy()) for a in acts]
        worst_layer, lp_o, lse_o = _oracle_from_inputs(cfg, tok, cu, sw, ads, xs, on)
        lp_err = max(np.abs(to_np(lp2[rows]) - lp_o).max(), np.abs(to_np(lse2[rows]) - lse_o).max())
        out[on] = (worst_layer, lp_err, torch.from_numpy(lp_o))
    return out


def _rounding_floor(cfg, tok, cu, mask, sw, ads, want):
    """How far the oracle's own step moves when it accumulates in fp32 instead of fp64
    (same bf16 storage points): the spread rounding alone puts on the free-running
    loss and gradients.  Returns (relative loss spread, normwise gradient spread).

    The loss spread is twice that single fp32 draw, or for DPO three standard
    deviations of the loss under rounding if larger.  A DPO loss is a function of each
    pair's margin, a sum of per-token policy - reference logprob differences, so one
    draw of it says little about its spread (the same draw measured 1.4% and 2.6% on two
    hosts whose fp32 matrix products differ).  The per-token differences e_t of the two
    oracle runs estimate it from every response position: with s_e their standard
    deviation, a pair's margin moves by s_e sqrt(n_c + n_r) and the loss, the mean over
    pairs of softplus(-beta z_p), by beta / npairs * sqrt(sum_p sigmoid(-z_p)^2
    (n_c + n_r)) * s_e.  A Gaussian draw beyond three of those has probability 0.3%."""
    with om.accumulate_in(torch.float32):
        o32 = om.train_step(tok, cu, mask, om.cast_stack(sw, torch.float32), om.cast_adapters(ads, torch.float32),
                            cfg)
    l64 = float(want["loss"])
    spread = 2 * abs(float(o32["loss"]) - l64) / abs(l64)
    if cfg.method == "dpo":
        m = np.asarray(mask, bool)
        e = (o32["lp"].double().numpy() - want["lp"].numpy()) - (o32["lp_ref"].double().numpy() - want["lp_ref"].numpy())
        s_e = float(e[m].std())
        n = np.array([int(m[cu[i]:cu[i + 1]].sum()) for i in range(len(cu) - 1)], np.float64)
        margin = want["pi"].numpy() - want["ref"].numpy()
        z = cfg.beta * (margin[0::2] - margin[1::2])
        sig = 1.0 / (1.0 + np.exp(z))
        s_loss = cfg.beta / len(z) * np.sqrt(np.sum(sig ** 2 * (n[0::2] + n[1::2]))) * s_e
        spread = max(spread, 3 * s_loss / abs(l64))
    g64 = np.concatenate([x.numpy().ravel() for layer in want["grads"] for x in layer])
    g32 = np.concatenate([x.double().numpy().ravel() for layer in o32["grads"] for x in layer])
    return spread, rel_err(g32, g64)


@pytest.mark.parametrize("cfg,vrows,cu,free_lp", PARITY, ids=[p[0].name for p in PARITY])
def test_step_matches_oracle(cfg, vrows, cu, free_lp):
    tok, cu, mask = _batch(cfg, 0, cu)
    nseq = len(cu) - 1
    st = _stack(cfg, vocab_chunk_rows=vrows, max_tokens=int(cu[-1]), max_seqs=nseq,
                max_seq_len=int(np.diff(cu).max()))
    shared = cfg.method == "dpo" and st.shared_read
    if shared:
        st.capture_reference()
    o, g, lp2, lse2 = _gpu_step(st, cfg, tok, cu, mask)
    sw = om.build_stack(cfg, 0, synth)
    ads = om.build_adapters(cfg, 0, synth)
    # 1. stage by stage: every layer and the vocabulary head from the GPU's own input, for
    #    the very forward whose loss is graded (the shared-read sweep when the step used it)
    lps, lps_o = {}, {}
    if shared:
        T = len(tok)
        for on, (worst_layer, lp_err, lo) in _teacher_forced_shared(st, cfg, tok, cu, sw, ads, lp2, lse2).items():
            assert worst_layer <= TOL_GRAD, (on, worst_layer)
            assert lp_err <= TOL_LP, (on, lp_err)
            lps[on], lps_o[on] = (lp2[:T] if on else lp2[T:]), lo
    else:
        for on in ([True, False] if cfg.method == "dpo" else [True]):
            worst_layer, lp_err, lps[on], lps_o[on] = _teacher_forced(st, cfg, tok, cu, mask, sw, ads, on)
            assert worst_layer <= TOL_GRAD, (on, worst_layer)
            assert lp_err <= TOL_LP, (on, lp_err)
    st.close()
    # the loss from those logprobs (policy sums, reference sums, DPO / SFT)
    if cfg.method == "dpo":
        pi_o, ref_o = om.seq_sums(lps_o[True], mask, cu), om.seq_sums(lps_o[False], mask, cu)
        loss_tf = float(om.dpo_loss(pi_o, ref_o, cfg.beta))
        # the DPO margin of each sequence, pi - ref, is a small difference of two large
        # sums: check it directly (absolute), not only through the loss near ln 2.  From
        # the same last hidden states only the vocabulary head differs (fp32 against fp64
        # accumulation, about 2e-5 per token); 1e-4 per summed position leaves 5x room.
        count = max(int(mask[cu[i]:cu[i + 1]].sum()) for i in range(nseq))
        m_gpu = to_np(o["pi"]) - to_np(o["ref"])
        m_o = np.asarray(pi_o, np.float64) - np.asarray(ref_o, np.float64)
        assert np.abs(m_gpu - m_o).max() <= 1e-4 * count, (m_gpu, m_o)
    else:
        loss_tf = float(om.sft_loss(lps_o[True], mask))
    assert abs(o["loss"].item() - loss_tf) <= TOL_LOSS * abs(loss_tf), (o["loss"].item(), loss_tf)
    # 2. the whole step free-running: bounded by the stated tolerance or, where bf16
    #    storage rounding alone moves the oracle further, by that measured spread
    #    (twice the gradients' fp32 draw; the loss spread as _rounding_floor derives it)
    want = om.train_step(tok, cu, mask, sw, ads, cfg)
    gflat = np.concatenate([x.numpy().ravel() for layer in want["grads"] for x in layer])
    floor_loss, floor_grad = _rounding_floor(cfg, tok, cu, mask, sw, ads, want)
    tol_loss, tol_grad = max(TOL_LOSS, floor_loss), max(TOL_GRAD, 2 * floor_grad)
    assert abs(o["loss"].item() - float(want["loss"])) <= tol_loss * abs(float(want["loss"])), (floor_loss,)
    assert rel_err(to_np(g), gflat) <= tol_grad, (floor_grad,)
    if free_lp:
        assert np.abs(to_np(lps[True]) - want["lp"].numpy()).max() <= TOL_LP
        if cfg.method == "dpo":
            assert np.abs(to_np(lps[False]) - want["lp_ref"].numpy()).max() <= TOL_LP
    if cfg.method == "dpo":
        # a sequence sum adds up to `count` per-token logprobs
        assert np.abs(to_np(o["pi"]) - want["pi"].numpy()).max() <= TOL_LP * count
        assert np.abs(to_np(o["ref"]) - want["ref"].numpy()).max() <= TOL_LP * count


# ------------------------------------------------------------------ invariants

def _run_all(st, cfg, tok, cu, mask):
    o, g, lp_ref, lse_ref = _gpu_step(st, cfg, tok, cu, mask)
    t, c, m = st.upload_batch(tok, cu, mask)
    st.fwd(t, c, m, adapter_on=True, save=False)
    lp_pol, _ = st.logprobs(len(tok))
    assert st.sync(300000) == 0
    return {k: v.clone() for k, v in o.items()}, g, lp_ref, lp_pol


@pytest.mark.parametrize("vrows", [256, 0])
def test_streamed_equals_resident_bit_exact(vrows):
    cfg = SMALL_DPO
    tok, cu, mask = _batch(cfg)
    a = _stack(cfg, resident=False, vocab_chunk_rows=vrows)
    b = _stack(cfg, resident=True, vocab_chunk_rows=vrows)
    ra = _run_all(a, cfg, tok, cu, mask)
    rb = _run_all(b, cfg, tok, cu, mask)
    sa, sb = a.stats(), b.stats()
    a.close()
    b.close()
    for x, y in zip(ra[1:], rb[1:]):
        assert torch.equal(x, y)
    for k in ("pi", "ref", "loss", "coeffs"):
        assert torch.equal(ra[0][k], rb[0][k]), k
    # the streamed context really streamed (a shared-read DPO step and one more forward
    # sweep, less the layers still in a slot at each turnaround); the resident one read
    # each layer once
    assert sa["layer_reads"] >= 2 * cfg.layers
    assert sb["layer_reads"] == cfg.layers


def _one_and_two(cfg):
    two = _stack(cfg, dpo_shared_read=False)
    one = L.Stack(cfg, device="cuda:0", dpo_shared_read=True)
    one.adopt_base(two)
    one.set_adapters_synthetic(synth, 0)
    assert one.shared_read and not two.shared_read
    return one, two


def test_shared_read_dpo_equals_two_passes():
    """Policy and reference forward in one sweep of the streamed layers give the very
    sums, loss, coefficients, logprobs and gradients of two separate sweeps, bit for bit,
    with 2 instead of 3 layer reads.  Every product of this stack runs whole tiles (each
    output summed in k order, whatever the tile shape), and every other kernel is
    row-independent, so the doubled batch changes nothing a row computes."""
    cfg = SMALL_DPO
    tok, cu, mask = _batch(cfg)
    one, two = _one_and_two(cfg)
    res, reads = {}, {}
    for name, st in (("two", two), ("one", one)):
        st.stats(reset=True)
        o, g, lp, _ = _gpu_step(st, cfg, tok, cu, mask)
        reads[name] = st.stats()["layer_reads"]
        res[name] = ({k: v.clone() for k, v in o.items()}, g, lp)
    one.close()
    two.close()
    (o2, g2, lp2), (o1, g1, lp1) = res["two"], res["one"]
    T = len(tok)
    # the two-pass form leaves the reference pass as its last forward
    assert torch.equal(lp1[T:], lp2)
    for k in ("pi", "ref", "loss", "coeffs"):
        assert torch.equal(o1[k], o2[k]), k
    assert torch.equal(g1, g2)
    assert reads["two"] >= 3 * cfg.layers - 2 and reads["one"] <= 2 * cfg.layers


def test_shared_read_dpo_8b_width_layers_match_two_passes():
    """At the Llama-3.1-8B widths the one-sweep products have twice the rows and take the
    paired split-tile schedule, so their fp32 sums run in another order than the T-row
    products of two sweeps: the forms agree to rounding, not bit for bit.  Both halves of
    the first decoder layer start from bit-identical embeddings, so their outputs must
    agree within the layer bound (each is within it of the exact layer); the last
    layer's are checked against the oracle by test_step_matches_oracle.  The read
    counts: 2 L against 3 L."""
    cfg = synth.small_stack(synth.LLAMA_8B, layers=2, vocab=8192, seq_len=512, nseq=2, prompt_len=256)
    tok, cu, mask = _batch(cfg)
    T, H = len(tok), cfg.hidden
    one, two = _one_and_two(cfg)
    one.capture_reference()
    reads = {}
    for name, st in (("two", two), ("one", one)):
        st.stats(reset=True)
        _gpu_step(st, cfg, tok, cu, mask)
        reads[name] = st.stats()["layer_reads"]
    pol1 = one.activation(1, T)
    ref1 = one.ref_capture[T * H: 2 * T * H].view(T, H).clone()
    assert one.sync(300000) == 0
    t_, c_, m_ = two.upload_batch(tok, cu, mask)
    outs = {}
    for on in (True, False):
        two.fwd(t_, c_, m_, adapter_on=on, save=True)
        outs[on] = two.activation(1, T)
    assert two.sync(300000) == 0
    one.close()
    two.close()
    assert rel_err(to_np(pol1), to_np(outs[True])) <= TOL_GRAD
    assert rel_err(to_np(ref1), to_np(outs[False])) <= TOL_GRAD
    assert not torch.equal(pol1, ref1)    # the adapter moved the policy rows
    assert reads["two"] >= 3 * cfg.layers - 2 and reads["one"] <= 2 * cfg.layers


def test_repeat_step_is_deterministic():
    cfg = SMALL_DPO
    tok, cu, mask = _batch(cfg)
    st = _stack(cfg, vocab_chunk_rows=256)
    r1 = _run_all(st, cfg, tok, cu, mask)
    r2 = _run_all(st, cfg, tok, cu, mask)
    st.close()
    for x, y in zip(r1[1:], r2[1:]):
        assert torch.equal(x, y)
    assert torch.equal(r1[0]["loss"], r2[0]["loss"])


def test_adapter_off_equals_base_and_zero_b():
    cfg = SMALL_DPO
    tok, cu, mask = _batch(cfg)
    base = _stack(cfg, adapters=False)
    zb = _stack(cfg, zero_b=True)
    on = _stack(cfg)
    t, c, m = base.upload_batch(tok, cu, mask)
    base.fwd(t, c, m, adapter_on=True, save=False)
    lp_base, lse_base = base.logprobs(len(tok))
    res = {}
    for name, st in (("zb", zb), ("on", on)):
        t2, c2, m2 = st.upload_batch(tok, cu, mask)
        st.fwd(t2, c2, m2, adapter_on=False, save=False)
        res[name + "_off"] = st.logprobs(len(tok))[0]
        st.fwd(t2, c2, m2, adapter_on=True, save=False)
        res[name + "_on"] = st.logprobs(len(tok))[0]
    for st in (base, zb, on):
        assert st.sync(60000) == 0
        st.close()
    assert torch.equal(res["on_off"], lp_base)      # reference pass = frozen base
    assert torch.equal(res["zb_off"], lp_base)
    assert torch.equal(res["zb_on"], lp_base)       # B = 0 adds exact zeros
    assert not torch.equal(res["on_on"], lp_base)   # a real adapter changes the policy


def test_dpo_loss_is_ln2_at_policy_equals_reference():
    cfg = SMALL_DPO
    tok, cu, mask = _batch(cfg)
    st = _stack(cfg, zero_b=True)
    o, g, _, _ = _gpu_step(st, cfg, tok, cu, mask)
    st.close()
    assert torch.equal(o["pi"], o["ref"])
    assert o["loss"].item() == pytest.approx(math.log(2.0), rel=1e-6)
    # dL/dB = -beta sigma(0) ... != 0 while dL/dA = 0 exactly (B = 0 blocks it)
    gn = to_np(g)
    r, H = cfg.lora_r, cfg.hidden
    per = 2 * r * H + r * (cfg.n_q + cfg.n_kv)
    for l in range(cfg.layers):
        blk = gn[l * per:(l + 1) * per]
        a_q = blk[: r * H]
        b_q = blk[r * H: r * H + cfg.n_q * r]
        assert np.all(a_q == 0.0)
        assert np.abs(b_q).max() > 0.0


def test_sft_loss_counts_and_sequence_sums():
    cfg = SMALL_DPO.with_(name="tiny-sft", method="sft", prompt_len=0)
    tok, cu, mask = _batch(cfg)
    st = _stack(cfg)
    o, _, lp, _ = _gpu_step(st, cfg, tok, cu, mask)
    st.close()
    lpn = to_np(lp)
    sums = [lpn[cu[i]:cu[i + 1]][mask[cu[i]:cu[i + 1]] > 0].sum() for i in range(cfg.nseq)]
    assert np.allclose(to_np(o["sums"]), sums, rtol=1e-5, atol=1e-3)
    assert o["loss"].item() == pytest.approx(-sum(sums) / mask.sum(), rel=1e-5)
    # last position of every sequence has no target
    assert np.all(lpn[cu[1:] - 1] == 0.0)


def test_bounded_sync_gives_up_on_a_slow_copy():
    """A host-side delay in the copy path makes ls_sync's time limit run out (no GPU fault)."""
    cfg = SMALL_DPO
    tok, cu, mask = _batch(cfg)
    st = _stack(cfg)
    t, c, m = st.upload_batch(tok, cu, mask)
    assert st.sync(60000) == 0
    L.check(L.lib().ls_debug_copy_delay(st.ctx, 300), st.ctx)
    st.fwd(t, c, m, adapter_on=True, save=False)
    assert st.sync(50) == L.LS_ERR_TIMEOUT
    L.check(L.lib().ls_debug_copy_delay(st.ctx, 0), st.ctx)
    assert st.sync(120000) == 0
    st.close()


def test_state_errors_are_reported():
    cfg = SMALL_DPO
    st = _stack(cfg)
    coeffs = torch.zeros(cfg.nseq, dtype=torch.float32, device=DEV)
    rc = L.lib().stream_step_bwd(st.ctx, coeffs.data_ptr())
    assert rc == L.LS_ERR_STATE
    assert "no forward" in L.last_error(st.ctx)
    # errors are sticky on the context
    assert L.lib().lora_grads(st.ctx, None, 0) == L.LS_ERR_STATE
    st.close()


def test_unpinned_layer_memory_is_refused():
    cfg = SMALL_DPO
    st = L.Stack(cfg, device="cuda:0")
    buf = np.zeros(st.img_bytes, np.uint8)   # pageable host memory
    lh = L.ls_layer_host()
    base = buf.ctypes.data
    for i, n in enumerate(("q", "k", "v", "o", "gate", "up", "down")):
        setattr(lh, n, L.ls_nf4_host(base + st.offs[i], base + st.offs[7 + i]))
    lh.attn_norm = base + st.offs[14]
    lh.mlp_norm = base + st.offs[15]
    import ctypes as C
    rc = L.lib().load_layer_nf4(st.ctx, 0, C.byref(lh))
    assert rc == L.LS_ERR_ARG
    assert "not pinned" in L.last_error(st.ctx)
    st.close()


# ------------------------------------------------------------------ full sizes

def _full_size_sampled(cfg, sample_layers):
    """Run the stack's shared-read DPO forward in the bench's launch configuration and
    check sampled layers and vocabulary rows against the oracle, teacher-forced."""
    tok, cu, mask = _batch(cfg)
    st = _stack(cfg)
    t, c, m = st.upload_batch(tok, cu, mask)
    pi = torch.empty(cfg.nseq, dtype=torch.float32, device=DEV)
    ref = torch.empty_like(pi)
    st.fwd_dpo(t, c, m, pi, ref)
    lp, lse = st.logprobs()
    acts = {l: st.activation(l, len(tok)) for l in sample_layers + [l + 1 for l in sample_layers]}
    hL = st.activation(cfg.layers, len(tok))
    assert st.sync(300000) == 0, L.last_error(st.ctx)
    st.close()
    ads = om.build_adapters(cfg, 0, synth)
    with torch.no_grad():
        for l in sample_layers:
            w = {n: om.dequant_weight(synth.weight(cfg, l, n, 0)) for n in ("q", "k", "v", "o", "gate", "up", "down")}
            lw = om.LayerWeights(w["q"], w["k"], w["v"], w["o"], w["gate"], w["up"], w["down"],
                                 om.t64(synth.norm_weight(cfg, l, 0, 0)), om.t64(synth.norm_weight(cfg, l, 1, 0)))
            x = om.t64(acts[l].float().cpu().numpy())
            y = om.decoder_layer(x, lw, ads[l], cfg, cu, adapter_on=True)
            assert rel_err(to_np(acts[l + 1]), y.numpy()) <= TOL_GRAD, l
        rows = np.random.default_rng(3).choice(len(tok), 16, replace=False)
        head = om.dequant_weight(synth.weight(cfg, -1, "lm_head", 0))
        hf = om.rmsnorm(om.t64(hL.float().cpu().numpy()[rows]), om.t64(synth.norm_weight(cfg, -1, 0, 0)), cfg.eps)
        logits = hf @ head.T
        lse_o = torch.logsumexp(logits, dim=-1).numpy()
        y = om.targets(tok, cu)[rows]
        lp_o = np.where(y >= 0, logits.numpy()[np.arange(len(rows)), np.maximum(y, 0)] - lse_o, 0.0)
    # policy rows are the first T of the shared pass
    assert np.abs(to_np(lse)[rows] - lse_o).max() <= TOL_LP
    assert np.abs(to_np(lp)[rows] - lp_o).max() <= TOL_LP


@pytest.mark.slow
def test_llama8b_full_sampled_layers_and_vocab_match_oracle():
    """The full 32-layer Llama-3.1-8B-shaped stack in the bench's launch configuration
    (shared-read DPO forward over 2 x 512 tokens): layers 0, 15 and 31 recomputed by the
    oracle from the GPU's own stored input of each (normwise <= 1e-2), and the full
    128256-row vocabulary head on 16 sampled token rows from the GPU's final hidden
    state (per-token logprob and log-sum-exp <= 2e-2)."""
    _full_size_sampled(synth.LLAMA_8B, [0, 15, 31])


@pytest.mark.slow
def test_qwen32b_full_capped_sampled_layers_and_vocab_match_oracle():
    """The full 64-layer Qwen2.5-32B-shaped stack under its 4 GiB workspace cap
    (shared-read DPO forward over 2 x 1024 tokens): layers 0 and 63 and 16 rows of the
    152064-row vocabulary head against the oracle, teacher-forced, as above."""
    _full_size_sampled(synth.QWEN_32B, [0, 63])


@pytest.mark.slow
def test_llama8b_full_streamed_equals_resident_and_ln2():
    """The full 32-layer Llama-3.1-8B-shaped DPO step, in the bench's launch
    configuration: streamed = resident bit for bit; B = 0 gives ln 2."""
    cfg = synth.LLAMA_8B
    tok, cu, mask = _batch(cfg)
    a = _stack(cfg)
    ra = _run_all(a, cfg, tok, cu, mask)
    sa = a.stats()
    # same Stack, adapters with B = 0
    a.set_adapters_synthetic(synth, 0, zero_b=True)
    o0, _, _, _ = _gpu_step(a, cfg, tok, cu, mask)
    a.set_adapters_synthetic(synth, 0)
    b = L.Stack(cfg, device="cuda:0", resident=True)
    b.adopt_base(a)                          # the same pinned host images
    b.set_adapters_synthetic(synth, 0)
    rb = _run_all(b, cfg, tok, cu, mask)
    b.close()
    a.close()
    for x, y in zip(ra[1:], rb[1:]):
        assert torch.equal(x, y)
    assert torch.equal(ra[0]["loss"], rb[0]["loss"])
    assert np.isfinite(to_np(ra[1])).all() and np.abs(to_np(ra[1])).max() > 0
    assert o0["loss"].item() == pytest.approx(math.log(2.0), rel=1e-6)
    assert sa["layer_reads"] >= 2 * cfg.layers


def test_tiny_dpo_step_matches_golden():
    """The GPU step against the oracle-written fixture of tests/golden/ (same bounds)."""
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_dpo_step.json")))
    c = g["config"]
    cfg = synth.StackConfig("golden-tiny-dpo", **c)
    tok, cu, mask = _batch(cfg)
    st = _stack(cfg)
    o, grads, _, _ = _gpu_step(st, cfg, tok, cu, mask)
    st.close()
    assert abs(o["loss"].item() - g["loss"]) <= TOL_LOSS * abs(g["loss"])
    count = int(mask[: cu[1]].sum())
    assert np.abs(to_np(o["pi"]) - np.array(g["pi"])).max() <= TOL_LP * count
    gn = to_np(grads)
    r, H = cfg.lora_r, cfg.hidden
    sizes = [r * H, cfg.n_q * r, r * H, cfg.n_kv * r]
    off = 0
    for layer in range(cfg.layers):
        for i, n in enumerate(sizes):
            norm = np.linalg.norm(gn[off: off + n])
            assert norm == pytest.approx(g["grad_norms"][layer][i], rel=TOL_GRAD * 5)
            off += n


def test_adapter_export_import_round_trip(tmp_path):
    """An adapter written with canonical keys and read back into a fresh context gives
    the same policy logprobs bit for bit, and they differ from the base's (so the
    import is not a silent no-op)."""
    cfg = SMALL_DPO
    tok, cu, mask = _batch(cfg)
    a = _stack(cfg)
    path = str(tmp_path / "adapter.safetensors")
    keys = a.export_adapter(path)
    assert len(keys) == 4 * cfg.layers and not any(".inner." in k for k in keys)
    b = L.Stack(cfg, device="cuda:0")
    b.adopt_base(a)
    base = L.Stack(cfg, device="cuda:0")
    base.adopt_base(a)
    b.import_adapter(path)
    lps = []
    for st in (a, b, base):
        t, c, m = st.upload_batch(tok, cu, mask)
        st.fwd(t, c, m, adapter_on=True, save=False)
        lps.append(st.logprobs(len(tok))[0])
        assert st.sync(60000) == 0
    for st in (b, base, a):
        st.close()
    assert torch.equal(lps[0], lps[1])
    assert not torch.equal(lps[1], lps[2])


def test_adamw_step_matches_oracle():
    """Two AdamW steps on the bound adapters from the GPU's own gradients, against the
    oracle's AdamW applied to the same gradients (fp32 vs fp64); the bf16 factors the
    forward reads are the rounded master weights."""
    cfg = SMALL_DPO
    tok, cu, mask = _batch(cfg)
    st = _stack(cfg)
    st.init_optimizer(lr=1e-3, betas=(0.9, 0.99), eps=1e-8, weight_decay=0.1)
    p = torch.from_numpy(to_np(st.opt["master"]))
    m = torch.zeros_like(p)
    v = torch.zeros_like(p)
    for t in (1, 2):
        t_, c_, m_ = st.upload_batch(tok, cu, mask)
        st.dpo_step(t_, c_, m_, cfg.beta)
        g = st.grads(zero_after=False)
        st.optimizer_step(zero_grads=True)
        assert st.sync(60000) == 0, L.last_error(st.ctx)
        om.adamw_update(p, torch.from_numpy(to_np(g)), m, v, t, 1e-3, 0.9, 0.99, 1e-8, 0.1)
        assert rel_err(to_np(st.opt["master"]), p.numpy()) <= 1e-5
        assert float(torch.from_numpy(to_np(st.grads())).abs().max()) == 0.0     # cleared
    flat_bf16 = torch.cat([st.adapters[l][k].float().ravel() for l in range(cfg.layers)
                           for k in ("aq", "bq", "av", "bv")])
    assert torch.equal(flat_bf16, st.opt["master"].to(torch.bfloat16).float())
    st.close()


def _unflatten_adapters(cfg, flat: torch.Tensor):
    """Adapters (fp64, bf16-rounded as the forward reads them) from a flat vector in
    lora_grads' order: per layer A_q [r, H], B_q [nq, r], A_v [r, H], B_v [nkv, r]."""
    r, H = cfg.lora_r, cfg.hidden
    shapes = [(r, H), (cfg.n_q, r), (r, H), (cfg.n_kv, r)]
    out, o = [], 0
    for _ in range(cfg.layers):
        ts = []
        for sh in shapes:
            n = sh[0] * sh[1]
            ts.append(om.bf16r(flat[o:o + n].reshape(sh).clone()))
            o += n
        out.append(om.Adapter(*ts))
    return out


def test_adamw_trajectory_matches_oracle():
    """Five consecutive training steps (DPO forward, loss, backward, AdamW on the fp32
    master weights, bf16 factors for the next forward) against the oracle running the
    same loop on its own: loss and sequence sums at every step, master weights after
    every update.  Each step feeds the next, so a drift in any part of the step would
    grow across them.

    Adam's first update is lr times the sign of each gradient element, so an element
    whose gradient lies within rounding noise of zero may step the other way on the two
    sides (a 2 lr difference).  The master weights are therefore compared on the
    elements whose first gradient stands clear of that noise (|g| >= 0.1 max|g|; the
    gradients agree to 1e-2 of max|g|), and at most 5% of all elements may differ by
    more than lr / 2."""
    cfg = SMALL_DPO
    tok, cu, mask = _batch(cfg)
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.999, 1e-8, 0.01
    st = _stack(cfg)
    st.init_optimizer(lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd)
    sw = om.build_stack(cfg, 0, synth)
    ads = om.build_adapters(cfg, 0, synth)
    p = torch.cat([x.detach().ravel() for ad in ads for x in ad.params()])
    m, v = torch.zeros_like(p), torch.zeros_like(p)
    count = max(int(mask[cu[i]:cu[i + 1]].sum()) for i in range(cfg.nseq))
    losses = []
    for t in range(1, 6):
        t_, c_, m_ = st.upload_batch(tok, cu, mask)
        o = st.dpo_step(t_, c_, m_, cfg.beta)
        st.optimizer_step(zero_grads=True)
        assert st.sync(60000) == 0, L.last_error(st.ctx)
        want = om.train_step(tok, cu, mask, sw, ads, cfg)
        g = torch.cat([x.ravel() for layer in want["grads"] for x in layer])
        if t == 1:
            clear = (g.abs() >= 0.1 * g.abs().max()).numpy()
        om.adamw_update(p, g, m, v, t, lr, b1, b2, eps, wd)
        ads = _unflatten_adapters(cfg, p)
        loss, loss_o = o["loss"].item(), float(want["loss"])
        assert abs(loss - loss_o) <= TOL_LOSS * abs(loss_o), (t, loss, loss_o)
        assert np.abs(to_np(o["pi"]) - want["pi"].numpy()).max() <= TOL_LP * count, t
        assert np.abs(to_np(o["ref"]) - want["ref"].numpy()).max() <= TOL_LP * count, t
        mg, mo = to_np(st.opt["master"]), p.numpy()
        assert rel_err(mg[clear], mo[clear]) <= TOL_GRAD, t
        assert np.mean(np.abs(mg - mo) > 0.5 * lr) <= 0.05, t
        losses.append((loss, loss_o))
    st.close()
    # the loop trains: the loss falls on both sides
    assert losses[-1][0] < losses[0][0] and losses[-1][1] < losses[0][1]


def test_file_backed_layers_match_pinned_ram(tmp_path):
    """Layers streamed from a file through pinned staging buffers give the same step,
    bit for bit, as the same images held in pinned RAM; every layer read goes through
    the file."""
    cfg = SMALL_DPO
    tok, cu, mask = _batch(cfg)
    ram = _stack(cfg, vocab_chunk_rows=256)
    path = str(tmp_path / "layers.bin")
    ram.write_layer_file(path)
    disk = L.Stack(cfg, device="cuda:0", vocab_chunk_rows=256)
    disk.adopt_base(ram)
    disk.set_adapters_synthetic(synth, 0)
    disk.use_layer_file(path, nbuf=2)
    disk.stats(reset=True)
    r_ram = _run_all(ram, cfg, tok, cu, mask)
    r_disk = _run_all(disk, cfg, tok, cu, mask)
    st = disk.stats()
    ram.close()
    disk.close()
    for x, y in zip(r_ram[1:], r_disk[1:]):
        assert torch.equal(x, y)
    for k in ("pi", "ref", "loss", "coeffs"):
        assert torch.equal(r_ram[0][k], r_disk[0][k]), k
    assert st["layer_reads"] >= 2 * cfg.layers
    assert st["file_bytes"] == st["layer_reads"] * disk.img_bytes


def test_layer_file_errors_are_reported(tmp_path):
    cfg = SMALL_DPO
    st = L.Stack(cfg, device="cuda:0")
    short = tmp_path / "short.bin"
    short.write_bytes(b"\0" * 1000)
    import ctypes as C
    assert L.lib().load_layer_file(st.ctx, 0, str(short).encode(), 0) == L.LS_ERR_ARG
    assert "shorter" in L.last_error(st.ctx)
    assert L.lib().load_layer_file(st.ctx, 0, str(tmp_path / "missing.bin").encode(), 0) == L.LS_ERR_ARG
    st.close()


def test_degenerate_inputs():
    """Empty batches and out-of-range sizes are refused on the host; a zero-row product
    launches nothing; single-token sequences (no next-token target) contribute zero
    logprob and the rest of the batch is unaffected."""
    import ctypes as C
    cfg = SMALL_DPO.with_(method="sft", prompt_len=0)
    st = _stack(cfg, max_tokens=cfg.tokens, max_seqs=6)
    tok, cu, mask = _batch(cfg)
    t, c, m = st.upload_batch(tok, cu, mask)
    sums = torch.empty(cfg.nseq, dtype=torch.float32, device=DEV)
    assert L.lib().stream_step_fwd(st.ctx, t.data_ptr(), 0, cfg.nseq, c.data_ptr(), m.data_ptr(), 1, 0,
                                   sums.data_ptr()) == L.LS_ERR_ARG
    st.close()
    st = _stack(cfg, max_tokens=cfg.tokens, max_seqs=6)
    assert L.lib().stream_step_fwd(st.ctx, t.data_ptr(), cfg.tokens + 1, cfg.nseq, c.data_ptr(), m.data_ptr(), 1, 0,
                                   sums.data_ptr()) == L.LS_ERR_ARG
    st.close()
    # single-token sequences next to a normal one
    st = _stack(cfg, max_tokens=cfg.tokens, max_seqs=6)
    cu1 = np.array([0, 1, 2, 50, 51], np.int32)
    tok1 = tok[:51]
    mask1 = np.ones(51, np.uint8)
    mask1[cu1[1:] - 1] = 0
    t1, c1, m1 = st.upload_batch(tok1, cu1, mask1)
    st.fwd(t1, c1, m1, adapter_on=True, save=False)
    lp1, _ = st.logprobs(51)
    cu2 = np.array([0, 48], np.int32)
    t2, c2, m2 = st.upload_batch(tok[2:50], cu2, np.ones(48, np.uint8))
    st.fwd(t2, c2, m2, adapter_on=True, save=False)
    lp2, _ = st.logprobs(48)
    assert st.sync(60000) == 0
    st.close()
    lp1n, lp2n = to_np(lp1), to_np(lp2)
    assert lp1n[0] == 0.0 and lp1n[1] == 0.0 and lp1n[50] == 0.0
    # the 48-token sequence gives the same logprobs wherever it sits in the batch
    np.testing.assert_array_equal(lp1n[2:50], lp2n)
    # zero-row product: nothing launched, output untouched
    w = synth.weight(cfg, 0, "q")
    pk, am = L.quantize_host(w)
    p, a = torch.from_numpy(pk).to(DEV), torch.from_numpy(am).to(DEV)
    out = torch.full((4, w.shape[0]), 7.0, dtype=torch.bfloat16, device=DEV)
    x = torch.zeros((4, w.shape[1]), dtype=torch.bfloat16, device=DEV)
    L.call("lsk_nf4_gemm", 0, x, w.shape[1], 0, p, a, w.shape[0], w.shape[1], None, None, 0, 0, out, w.shape[0], None,
           0, 0, 0, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
