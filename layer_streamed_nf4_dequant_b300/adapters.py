"""LoRA adapter export and load with canonical keys (safetensors layout).

The pages report two ways a streamed adapter went wrong on save / load:
- saved keys gained a wrapper segment (".inner."), so standard loaders matched none of
  them and silently fell back to the base model (Show HN: Fine-tune an 8B model on a 4 GB
  laptop GPU; axbrief.com, "Beyond Memory: The Layer Streaming Breakthrough", with a
  one-line key check; evermx.com summary);
- "a streamed adapter loading as a no-op" (Soup: Fine-Tune an 8B Model on a 4 GB GPU,
  "The Core Idea: Layer Streaming", caveats).

Files written here carry only the canonical PEFT-style names
    base_model.model.model.layers.{l}.self_attn.{q_proj|v_proj}.lora_{A|B}.weight
(A [r, in], B [out, r]), with the rank and scale in the metadata.  The loader refuses a
file whose keys do not match that set exactly, or whose shapes disagree, so that a
renamed or wrapped key can never turn into a silent no-op.

The container format is safetensors: an 8-byte little-endian header length, a JSON
header {name: {dtype, shape, data_offsets}}, then the raw little-endian tensor bytes.
"""
from __future__ import annotations

import json
import struct
from typing import Dict, List, Tuple

import numpy as np

PREFIX = "base_model.model.model.layers"
PROJS = ("q_proj", "v_proj")

_DT = {"F32": np.float32, "F64": np.float64, "BF16": np.uint16, "F16": np.float16, "I32": np.int32}
_DT_NAME = {np.dtype(np.float32): "F32", np.dtype(np.float64): "F64", np.dtype(np.float16): "F16",
            np.dtype(np.int32): "I32"}


class AdapterKeyError(ValueError):
    """The file's tensor names or shapes do not match the expected adapter."""


def canonical_key(layer: int, proj: str, factor: str) -> str:
    """e.g. base_model.model.model.layers.3.self_attn.q_proj.lora_A.weight"""
    if proj not in PROJS or factor not in ("A", "B"):
        raise ValueError(f"bad projection / factor {proj!r} {factor!r}")
    return f"{PREFIX}.{layer}.self_attn.{proj}.lora_{factor}.weight"


def expected_shapes(layers: int, hidden: int, n_q: int, n_kv: int, r: int) -> Dict[str, Tuple[int, int]]:
    out = {}
    for l in range(layers):
        out[canonical_key(l, "q_proj", "A")] = (r, hidden)
        out[canonical_key(l, "q_proj", "B")] = (n_q, r)
        out[canonical_key(l, "v_proj", "A")] = (r, hidden)
        out[canonical_key(l, "v_proj", "B")] = (n_kv, r)
    return out


def write_safetensors(path: str, tensors: Dict[str, np.ndarray], metadata: Dict[str, str] | None = None,
                      bf16: Tuple[str, ...] = ()) -> None:
    """Write tensors; names in `bf16` hold uint16 bit patterns stored as BF16."""
    header: Dict[str, dict] = {}
    blobs: List[bytes] = []
    off = 0
    for name in sorted(tensors):
        a = np.ascontiguousarray(tensors[name])
        if name in bf16:
            if a.dtype != np.uint16:
                raise TypeError(f"{name}: bf16 tensors travel as uint16 bit patterns")
            dt = "BF16"
        else:
            dt = _DT_NAME[a.dtype]
        b = a.astype(a.dtype.newbyteorder("<"), copy=False).tobytes()
        header[name] = {"dtype": dt, "shape": list(a.shape), "data_offsets": [off, off + len(b)]}
        blobs.append(b)
        off += len(b)
    if metadata:
        header["__metadata__"] = {str(k): str(v) for k, v in metadata.items()}
    h = json.dumps(header, separators=(",", ":")).encode()
    h += b" " * ((8 - len(h) % 8) % 8)
    with open(path, "wb") as f:
        f.write(struct.pack("<Q", len(h)))
        f.write(h)
        for b in blobs:
            f.write(b)


def read_safetensors(path: str) -> Tuple[Dict[str, np.ndarray], Dict[str, str]]:
    """Tensors (BF16 as uint16 bit patterns) and the metadata of a safetensors file."""
    with open(path, "rb") as f:
        raw = f.read()
    (n,) = struct.unpack("<Q", raw[:8])
    header = json.loads(raw[8:8 + n])
    meta = header.pop("__metadata__", {})
    base = 8 + n
    out = {}
    for name, d in header.items():
        a, b = d["data_offsets"]
        arr = np.frombuffer(raw[base + a: base + b], dtype=np.dtype(_DT[d["dtype"]]).newbyteorder("<"))
        out[name] = arr.reshape(d["shape"]).copy()
    return out, meta


def save_adapter(path: str, adapters: List[Dict[str, np.ndarray]], lora_r: int, lora_alpha: float) -> List[str]:
    """adapters[l] = {"aq", "bq", "av", "bv"} as bf16 bit patterns (uint16); returns the keys."""
    tensors = {}
    for l, ad in enumerate(adapters):
        tensors[canonical_key(l, "q_proj", "A")] = ad["aq"]
        tensors[canonical_key(l, "q_proj", "B")] = ad["bq"]
        tensors[canonical_key(l, "v_proj", "A")] = ad["av"]
        tensors[canonical_key(l, "v_proj", "B")] = ad["bv"]
    write_safetensors(path, tensors, {"format": "pt", "lora_r": lora_r, "lora_alpha": lora_alpha,
                                      "target_modules": ",".join(PROJS)}, bf16=tuple(tensors))
    return sorted(tensors)


def load_adapter(path: str, layers: int, hidden: int, n_q: int, n_kv: int, r: int) -> List[Dict[str, np.ndarray]]:
    """Read an adapter file written with canonical keys; refuse anything else.

    Raises AdapterKeyError when a key is missing, unexpected (e.g. a wrapper segment
    such as ".inner." in its name) or has the wrong shape."""
    tensors, _ = read_safetensors(path)
    want = expected_shapes(layers, hidden, n_q, n_kv, r)
    missing = sorted(set(want) - set(tensors))
    extra = sorted(set(tensors) - set(want))
    if missing or extra:
        hint = ""
        if any(".inner." in k for k in extra):
            hint = " (keys carry a '.inner.' wrapper segment)"
        raise AdapterKeyError(f"adapter keys do not match{hint}: {len(missing)} missing (e.g. "
                              f"{missing[:1]}), {len(extra)} unexpected (e.g. {extra[:1]})")
    for k, shp in want.items():
        if tuple(tensors[k].shape) != shp:
            raise AdapterKeyError(f"{k}: shape {tuple(tensors[k].shape)}, expected {shp}")
    return [{"aq": tensors[canonical_key(l, "q_proj", "A")], "bq": tensors[canonical_key(l, "q_proj", "B")],
             "av": tensors[canonical_key(l, "v_proj", "A")], "bv": tensors[canonical_key(l, "v_proj", "B")]}
            for l in range(layers)]
