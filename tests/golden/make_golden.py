"""Write the oracle-generated regression fixtures of tests/golden/ (calls only oracle/ and synth/).

    python tests/golden/make_golden.py

tiny_dpo_step.json: one DPO step of a 2-layer, 256-wide stack (seed 0) -- loss, policy
and reference sequence sums, and the norm and first entries of every LoRA gradient --
computed by the fp64 oracle.  A later change to the oracle that moves these values must
say which passage of the pages (or which reading of it) justifies the move.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import synth  # noqa: E402
from oracle import model as om  # noqa: E402

TINY_DPO = synth.StackConfig("golden-tiny-dpo", layers=2, hidden=256, heads=4, kv_heads=2, head_dim=64, inter=512,
                             vocab=512, tied=False, rope_theta=1e4, eps=1e-6, lora_r=8, lora_alpha=16.0,
                             seq_len=48, nseq=2, prompt_len=16, method="dpo", beta=0.1)


def tiny_dpo_step():
    cfg = TINY_DPO
    tok, cu, mask = synth.tokens(cfg), synth.seq_offsets(cfg), synth.loss_mask(cfg)
    o = om.train_step(tok, cu, mask, om.build_stack(cfg, 0, synth), om.build_adapters(cfg, 0, synth), cfg)
    grads = [[g.numpy() for g in layer] for layer in o["grads"]]
    return {
        "config": {k: getattr(cfg, k) for k in ("layers", "hidden", "heads", "kv_heads", "head_dim", "inter",
                                                 "vocab", "tied", "rope_theta", "eps", "lora_r", "lora_alpha",
                                                 "seq_len", "nseq", "prompt_len", "method", "beta")},
        "seed": 0,
        "loss": float(o["loss"]),
        "pi": [float(x) for x in o["pi"]],
        "ref": [float(x) for x in o["ref"]],
        "grad_norms": [[float(np.linalg.norm(g)) for g in layer] for layer in grads],
        "grad_head": [[[float(v) for v in g.ravel()[:4]] for g in layer] for layer in grads],
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_dpo_step.json"), "w") as f:
        json.dump(tiny_dpo_step(), f, indent=1)
    print("wrote tiny_dpo_step.json")
