"""Adapter files with canonical keys (no GPU): round trip, and refusal of the key
mismatches the pages report (".inner." wrapper segments; an adapter that would load
as a silent no-op)."""
import json
import struct

import numpy as np
import pytest

from layer_streamed_nf4_dequant_b300 import adapters as A


def _ads(layers=2, H=64, nq=64, nkv=32, r=4, seed=0):
    rng = np.random.default_rng(seed)
    mk = lambda *s: rng.integers(0, 65535, s, dtype=np.uint16)
    return [{"aq": mk(r, H), "bq": mk(nq, r), "av": mk(r, H), "bv": mk(nkv, r)} for _ in range(layers)]


def test_round_trip_and_canonical_keys(tmp_path):
    ads = _ads()
    p = str(tmp_path / "adapter.safetensors")
    keys = A.save_adapter(p, ads, 4, 8.0)
    assert all(k.startswith("base_model.model.model.layers.") and ".inner." not in k for k in keys)
    assert "base_model.model.model.layers.1.self_attn.v_proj.lora_B.weight" in keys
    back = A.load_adapter(p, 2, 64, 64, 32, 4)
    for a, b in zip(ads, back):
        for k in a:
            np.testing.assert_array_equal(a[k], b[k])
    # the header is plain safetensors: 8-byte length, JSON, BF16 entries with offsets
    raw = open(p, "rb").read()
    (n,) = struct.unpack("<Q", raw[:8])
    hdr = json.loads(raw[8:8 + n])
    assert hdr["__metadata__"]["lora_r"] == "4"
    e = hdr["base_model.model.model.layers.0.self_attn.q_proj.lora_A.weight"]
    assert e["dtype"] == "BF16" and e["shape"] == [4, 64] and e["data_offsets"][1] - e["data_offsets"][0] == 4 * 64 * 2


def test_wrapped_keys_are_refused(tmp_path):
    ads = _ads()
    t = {}
    for l, ad in enumerate(ads):
        for proj, fa, fb in (("q_proj", "aq", "bq"), ("v_proj", "av", "bv")):
            t[f"base_model.model.model.layers.{l}.self_attn.{proj}.inner.lora_A.weight"] = ad[fa]
            t[f"base_model.model.model.layers.{l}.self_attn.{proj}.inner.lora_B.weight"] = ad[fb]
    p = str(tmp_path / "wrapped.safetensors")
    A.write_safetensors(p, t, bf16=tuple(t))
    with pytest.raises(A.AdapterKeyError, match="inner"):
        A.load_adapter(p, 2, 64, 64, 32, 4)


def test_missing_layers_and_wrong_shapes_are_refused(tmp_path):
    p = str(tmp_path / "a.safetensors")
    A.save_adapter(p, _ads(layers=1), 4, 8.0)
    with pytest.raises(A.AdapterKeyError, match="missing"):
        A.load_adapter(p, 2, 64, 64, 32, 4)
    A.save_adapter(p, _ads(layers=2, r=8), 8, 16.0)
    with pytest.raises(A.AdapterKeyError, match="shape"):
        A.load_adapter(p, 2, 64, 64, 32, 4)
