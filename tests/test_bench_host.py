"""Host-side logic of bench.py (no GPU): the per-step roofline model and the
max-over-ranks timing of a multi-process run (gloo, world size 2)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench
import synth


def _roof(s, reads_l, reads_v, shared, tflops, link, nvch=4, layer_b=122.7e6):
    vb = s.vocab * s.hidden * 0.5625 / nvch
    k = {"layer_reads": reads_l, "vocab_reads": reads_v, "h2d_bytes": reads_l * layer_b + reads_v * vb}
    return bench.link_roofline_ms(s, s.tokens, s.seq_len, s.nseq, k, layer_b, vb, nvch, tflops, link, shared), vb


def test_step_roofline_is_link_bound_for_a_slow_link():
    s = synth.LLAMA_8B
    layer_b = 122.7e6
    # two forward sweeps and the backward, every use a copy, all at 1 GB/s
    r, vb = _roof(s, 3 * s.layers, 3 * 4, False, tflops=1e9, link=1.0, layer_b=layer_b)
    want = (3 * s.layers * layer_b + 3 * 4 * vb) / 1e9 * 1e3
    assert r["ms"] == pytest.approx(want, rel=1e-9)
    assert r["link_ms"] == pytest.approx(want, rel=1e-9)


def test_step_roofline_shared_read_saves_one_sweep():
    s = synth.LLAMA_8B
    layer_b = 122.7e6
    two, vb = _roof(s, 3 * s.layers, 12, False, 1e9, 1.0, layer_b=layer_b)
    one, _ = _roof(s, 2 * s.layers, 8, True, 1e9, 1.0, layer_b=layer_b)
    assert two["ms"] - one["ms"] == pytest.approx((s.layers * layer_b + 4 * vb) / 1e9 * 1e3, rel=1e-9)
    assert one["flop"] == pytest.approx(two["flop"], rel=1e-12)


def test_step_roofline_reuse_saves_the_copy_not_the_compute():
    """An item still in a slot at the turnaround costs its FLOPs, not its bytes."""
    s = synth.LLAMA_8B
    full, vb = _roof(s, 2 * s.layers, 8, True, 1000.0, 50.0)
    reuse, _ = _roof(s, 2 * s.layers - 2, 6, True, 1000.0, 50.0)
    saved = full["ms"] - reuse["ms"]
    assert 0 < saved < (2 * 122.7e6 + 2 * vb) / 50e9 * 1e3
    # and the bound never exceeds the bytes moved at the link rate plus all compute at peak
    assert reuse["ms"] <= reuse["link_ms"] + reuse["compute_ms"]
    assert reuse["ms"] >= max(reuse["link_ms"], reuse["compute_ms"]) - 1e-9


def test_step_roofline_is_tensor_bound_for_an_infinite_link():
    s = synth.QWEN_3B.with_(method="sft")
    nvch = 2
    vb = s.vocab * s.hidden * 0.5625 / nvch
    k = {"layer_reads": 2 * s.layers, "vocab_reads": 2 * nvch, "h2d_bytes": 0.0}
    r = bench.link_roofline_ms(s, s.tokens, s.seq_len, s.nseq, k, 43.4e6, vb, nvch, 1000.0, 1e12, False)
    assert r["ms"] == pytest.approx(r["flop"] / 1e15 * 1e3, rel=1e-6)
    # forward 2 T P per layer dominates: the step is at least 4 T P L FLOPs (fwd + dX)
    assert r["flop"] >= 4 * s.tokens * bench.layer_params(s) * s.layers


def test_pcie_spec_rates():
    assert bench.pcie_spec_gbs(5, 16) == pytest.approx(63.02, rel=1e-3)
    assert bench.pcie_spec_gbs(6, 16) == pytest.approx(121.0, rel=1e-3)
    assert bench.pcie_spec_gbs(4, 8) == pytest.approx(15.75, rel=1e-3)


def test_layer_params_match_the_8b_shape():
    # q/k/v/o + gate/up/down of one Llama-3.1-8B layer: 218.1M weights
    assert bench.layer_params(synth.LLAMA_8B) == 218_103_808


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    bench.init_dist(ws, "gloo")
    got = bench.max_over_ranks(10.0 + rank, ws)
    bench.barrier(ws)
    q.put((rank, got))
    torch.distributed.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 11.0, 1: 11.0}


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the CPU oracle arm, run here on the small 896-wide
    config) prints one JSON line with every key of the bench contract."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--config", "layer-896",
                        "--steps", "1", "--warmup", "3"], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] >= 3 and d["ms_per_step"] > 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["dtype"] == "f64" and d["data"] == "synthetic" and d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
