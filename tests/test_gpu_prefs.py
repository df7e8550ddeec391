"""SimPO, ORPO and KTO on the GPU against the oracle (GPU required).

The pages list these preference losses beside DPO as methods run over the streamed
base (axbrief.com, "The Architecture of Low-VRAM Alignment"; evermx.com summary);
their formulas are the methods' own (see oracle/model.py).  The loss kernels are
checked against the oracle's autograd on given sequence sums (fp32 vs fp64: 1e-5
relative), and one whole streamed step of each method on a small stack against the
oracle's step (loss 1e-2 relative, LoRA gradients 1e-2 normwise).
"""
import numpy as np
import pytest
import torch

import layer_streamed_nf4_dequant_b300 as L
import synth
from oracle import model as om

from gpu_util import DEV, rel_err, to_np

pytestmark = pytest.mark.gpu

SMALL = synth.StackConfig("tiny-pref", layers=3, hidden=256, heads=4, kv_heads=2, head_dim=64, inter=512,
                          vocab=1024, tied=False, rope_theta=1e4, eps=1e-6, lora_r=16, lora_alpha=32.0,
                          seq_len=96, nseq=4, prompt_len=40, method="simpo", beta=2.0, simpo_gamma=0.5,
                          orpo_lambda=0.2, kto_lambda_d=1.0, kto_lambda_u=1.5)


def _sums_case(nseq, seed):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(rng.integers(20, 60, nseq))]).astype(np.int32)
    mask = (rng.random(cu[-1]) < 0.7).astype(np.uint8)
    counts = np.array([mask[cu[i]:cu[i + 1]].sum() for i in range(nseq)], np.float64)
    pi = (-counts * rng.uniform(1.0, 4.0, nseq)).astype(np.float32)
    ref = (pi + rng.normal(0, 2.0, nseq)).astype(np.float32)
    return cu, mask, pi, ref


def _run_loss(fn, *args):
    st = L.Stack(SMALL.with_(layers=1), device="cuda:0")
    loss = torch.empty(1, dtype=torch.float32, device=DEV)
    coeffs = torch.empty(len(args[0]), dtype=torch.float32, device=DEV)
    dev = [torch.from_numpy(a).to(DEV) if isinstance(a, np.ndarray) else a for a in args]
    rest = [a.data_ptr() if isinstance(a, torch.Tensor) else a for a in dev]
    L.check(getattr(L.lib(), fn)(st.ctx, *rest, loss.data_ptr(), coeffs.data_ptr()), st.ctx)
    assert st.sync(60000) == 0
    st.close()
    return loss.item(), to_np(coeffs)


@pytest.mark.parametrize("seed", [0, 1])
def test_simpo_orpo_kto_kernels_match_oracle(seed):
    nseq = 6
    cu, mask, pi, ref = _sums_case(nseq, seed)
    counts = om.seq_counts(mask, cu)
    # SimPO
    P = torch.from_numpy(pi.astype(np.float64)).requires_grad_(True)
    want = om.simpo_loss(P, counts, 2.0, 0.5)
    want.backward()
    loss, co = _run_loss("simpo_loss", pi, cu, mask, nseq // 2, 2.0, 0.5)
    assert loss == pytest.approx(float(want.detach()), rel=1e-5)
    np.testing.assert_allclose(co, P.grad.numpy(), rtol=1e-4, atol=1e-7)
    # ORPO
    P = torch.from_numpy(pi.astype(np.float64)).requires_grad_(True)
    want = om.orpo_loss(P, counts, 0.2)
    want.backward()
    loss, co = _run_loss("orpo_loss", pi, cu, mask, nseq // 2, 0.2)
    assert loss == pytest.approx(float(want.detach()), rel=1e-5)
    np.testing.assert_allclose(co, P.grad.numpy(), rtol=1e-4, atol=1e-7)
    # KTO, explicit labels
    des = np.array([1, 0, 1, 1, 0, 0], np.uint8)
    P = torch.from_numpy(pi.astype(np.float64)).requires_grad_(True)
    want = om.kto_loss(P, torch.from_numpy(ref.astype(np.float64)), torch.from_numpy(des), 0.1, 1.0, 1.5)
    want.backward()
    loss, co = _run_loss("kto_loss", pi, ref, des, nseq, 0.1, 1.0, 1.5)
    assert loss == pytest.approx(float(want.detach()), rel=1e-5)
    np.testing.assert_allclose(co, P.grad.numpy(), rtol=1e-4, atol=1e-8)


@pytest.mark.parametrize("method", ["simpo", "orpo", "kto"])
def test_streamed_preference_step_matches_oracle(method):
    cfg = SMALL.with_(method=method, beta=2.0 if method == "simpo" else 0.1)
    tok, cu, mask = synth.tokens(cfg), synth.seq_offsets(cfg), synth.loss_mask(cfg)
    st = L.Stack(cfg, device="cuda:0", vocab_chunk_rows=256)
    st.load_synthetic(synth, 0)
    st.set_adapters_synthetic(synth, 0)
    assert st.shared_read == (method == "kto")
    st.stats(reset=True)
    t, c, m = st.upload_batch(tok, cu, mask)
    o = st.pref_step(method, t, c, m)
    g = st.grads(zero_after=True)
    assert st.sync(120000) == 0, L.last_error(st.ctx)
    reads = st.stats()["layer_reads"]
    st.close()
    want = om.train_step(tok, cu, mask, om.build_stack(cfg, 0, synth), om.build_adapters(cfg, 0, synth), cfg)
    gflat = np.concatenate([x.numpy().ravel() for layer in want["grads"] for x in layer])
    assert abs(o["loss"].item() - float(want["loss"])) <= 1e-2 * abs(float(want["loss"]))
    assert rel_err(to_np(g), gflat) <= 1e-2
    # reference-free methods stream each layer for the policy forward and the backward only
    assert reads <= 2 * cfg.layers
