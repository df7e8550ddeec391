"""CPU oracle for layer-streamed NF4 LoRA fine-tuning — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The CUDA library never calls it, and it
shares no code with the CUDA library: the two meet only through the seeded
inputs of ``synth``.

What it computes is the plain, non-streamed definition of one training step of
the method the Soup pages describe: a frozen NF4 base ("Optionally quantizing
that streamed base to NF4", Soup: Fine-Tune an 8B Model on a 4 GB GPU, "The Core
Idea: Layer Streaming"), a plain LoRA on q_proj/v_proj with r = 16 (same page,
the soup.yaml listing), SFT next-token loss, and DPO whose reference logprobs come
from the same base with the adapter switched off (Show HN: Fine-tune an 8B model
on a 4 GB laptop GPU, opening paragraph).  Streaming changes where the weights
live, not what is computed, and the pages call the streamed result bit-exact
against a resident run (axbrief.com, "Beyond Memory: The Layer Streaming
Breakthrough"), so the oracle is simply the resident computation.

Precision: fp64 arithmetic (torch CPU float64), with bf16 storage emulated at the
tensor boundaries where the GPU path stores bf16.  Gradients come from autograd
through that fp64 graph (bf16 rounding passes gradients straight through).

Pins: every function here is checked against something other than itself in
``tests/test_oracle_pins.py`` (closed forms, invariants, brute force, finite
differences, library special cases).  Parity unpinned: none.
"""
from .nf4 import (NF4_TABLE, bf16_round_f32, nf4_quantize, nf4_dequantize, nf4_pack,
                  nf4_unpack)
from . import model

__all__ = ["NF4_TABLE", "bf16_round_f32", "nf4_quantize", "nf4_dequantize", "nf4_pack",
           "nf4_unpack", "model"]
