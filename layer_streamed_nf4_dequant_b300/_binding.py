"""ctypes binding of libls.so: argument marshalling only, same names as the C ABI.

Every computation happens in the library's CUDA kernels; this module converts
Python ints / torch tensors to pointers and raises on a non-zero status.  It
fails loudly when the compiled library is missing; there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libls.so")
HEADERS = [os.path.join(os.path.dirname(_PKG), "include", h) for h in ("ls.h", "ls_kernels.h")]

LS_OK, LS_ERR_ARG, LS_ERR_CAP, LS_ERR_CUDA, LS_ERR_TIMEOUT, LS_ERR_STATE, LS_ERR_DEVICE = 0, -1, -2, -3, -4, -5, -6
ERR_NAMES = {0: "LS_OK", -1: "LS_ERR_ARG", -2: "LS_ERR_CAP", -3: "LS_ERR_CUDA", -4: "LS_ERR_TIMEOUT",
             -5: "LS_ERR_STATE", -6: "LS_ERR_DEVICE"}


class LSError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERR_NAMES.get(code, code)}: {msg}")
        self.code = code


class ls_config(C.Structure):
    _fields_ = [("layers", C.c_int32), ("hidden", C.c_int32), ("heads", C.c_int32), ("kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("inter", C.c_int32), ("vocab", C.c_int32), ("tied", C.c_int32),
                ("lora_r", C.c_int32), ("lora_scale", C.c_float), ("rope_theta", C.c_float), ("eps", C.c_float),
                ("max_tokens", C.c_int32), ("max_seqs", C.c_int32), ("max_seq_len", C.c_int32),
                ("vocab_chunk_rows", C.c_int32), ("resident", C.c_int32), ("dpo_shared_read", C.c_int32),
                ("cap_bytes", C.c_uint64)]


class ls_nf4_host(C.Structure):
    _fields_ = [("packed", C.c_void_p), ("absmax", C.c_void_p)]


class ls_layer_host(C.Structure):
    _fields_ = [(n, ls_nf4_host) for n in ("q", "k", "v", "o", "gate", "up", "down")] + [
        ("attn_norm", C.c_void_p), ("mlp_norm", C.c_void_p)]


class ls_vocab_host(C.Structure):
    _fields_ = [("embed", ls_nf4_host), ("lm_head", ls_nf4_host), ("final_norm", C.c_void_p)]


class ls_stats_t(C.Structure):
    _fields_ = [("layer_reads", C.c_uint64), ("vocab_reads", C.c_uint64), ("h2d_bytes", C.c_uint64),
                ("slot_reuses", C.c_uint64), ("workspace_bytes", C.c_uint64), ("slot_bytes", C.c_uint64),
                ("act_store_bytes", C.c_uint64), ("vocab_chunks", C.c_int32), ("vocab_chunk_rows", C.c_int32),
                ("kernel_launches", C.c_uint64), ("file_bytes", C.c_uint64), ("file_read_ms", C.c_double)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class lsk_gemm_plan(C.Structure):
    _fields_ = [("nacc", C.c_int32), ("bn", C.c_int32), ("tiles_m", C.c_int32), ("tiles_n", C.c_int32),
                ("ctas", C.c_int32), ("whole_per_cta", C.c_int32), ("k_iters", C.c_int32), ("pair_rows", C.c_int32),
                ("split_iters", C.c_int64)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class ls_profile_t(C.Structure):
    _fields_ = [("launches", C.c_uint64 * 5), ("ms", C.c_double * 5), ("flop", C.c_double * 5),
                ("bytes", C.c_double * 5)]

    CLASSES = ("gemm_fwd", "gemm_dx", "attn_fwd", "attn_bwd", "other")

    def as_dict(self):
        return {c: {"launches": int(self.launches[i]), "ms": self.ms[i], "flop": self.flop[i],
                    "bytes": self.bytes[i]} for i, c in enumerate(self.CLASSES)}


P, I32, I64, U64, F32 = C.c_void_p, C.c_int32, C.c_int64, C.c_uint64, C.c_float

_SIGS = {
    "ls_plan": [C.POINTER(ls_config), C.POINTER(U64)],
    "ls_layer_layout": [C.POINTER(ls_config), C.POINTER(U64), C.POINTER(U64)],
    "ls_create": [C.POINTER(ls_config), P, U64, P, P, C.POINTER(P)],
    "ls_destroy": [P],
    "nf4_quantize": [P, I64, I64, P, P, I32],
    "load_layer_nf4": [P, I32, C.POINTER(ls_layer_host)],
    "load_vocab_nf4": [P, C.POINTER(ls_vocab_host)],
    "load_layer_file": [P, I32, C.c_char_p, U64],
    "ls_set_staging": [P, P, U64, I32],
    "ls_set_adapter": [P, I32, P, P, P, P, P, P, P, P],
    "stream_step_fwd": [P, P, I32, I32, P, P, I32, I32, P],
    "stream_step_fwd_dpo": [P, P, I32, I32, P, P, P, P],
    "seq_logprobs": [P, P, P],
    "dpo_loss": [P, P, P, I32, F32, P, P],
    "sft_loss": [P, P, I32, F32, P, P],
    "simpo_loss": [P, P, P, P, I32, F32, F32, P, P],
    "orpo_loss": [P, P, P, P, I32, F32, P, P],
    "kto_loss": [P, P, P, P, I32, F32, F32, F32, P, P],
    "stream_step_bwd": [P, P],
    "lora_grads": [P, P, I32],
    "lora_params": [P, P],
    "lora_adamw": [P, P, P, P, I32, F32, F32, F32, F32, F32, I32],
    "ls_sync": [P, I32],
    "ls_stats": [P, C.POINTER(ls_stats_t), I32],
    "ls_debug_copy_delay": [P, I32],
    "ls_read_activation": [P, I32, P],
    "ls_capture_reference": [P, P, U64],
    "ls_profile": [P, I32],
    "ls_profile_read": [P, C.POINTER(ls_profile_t)],
    "lsk_nf4_dequant": [P, P, I64, I32, P, P],
    "lsk_nf4_gemm": [I32, P, I64, I32, P, P, I32, I32, P, P, I32, I32, P, I64, P, I64, I32, I32, P],
    "lsk_nf4_gemm_plan": [I32, I32, I32, I32, I32, I32, I32, I32, I32, I32, I32, C.POINTER(lsk_gemm_plan)],
    "lsk_nf4_gemm_sk": [I32, P, I64, I32, P, P, I32, I32, P, P, I32, I32, P, I64, P, I64, I32, I32, I32, I32, P, U64,
                        P],
    "lsk_rmsnorm_fwd": [P, P, P, P, I32, I32, F32, P],
    "lsk_rmsnorm_bwd": [P, P, P, P, P, P, I32, I32, I32, P],
    "ls_rope_table": [P, P, I32, I32, F32],
    "lsk_rope_fwd": [P, I64, P, P, P, I32, I32, I32, P],
    "lsk_rope_bwd_cast": [P, P, I64, P, P, P, I32, I32, I32, I32, P],
    "lsk_attn_fwd": [P, I64, P, I32, I32, I32, I32, I32, P, I64, P, I32, P],
    "lsk_attn_bwd": [P, I64, P, P, I64, P, P, I32, I32, I32, I32, I32, P, P, I64, I32, P, P],
    "lsk_swiglu_fwd": [P, P, I32, I32, P],
    "lsk_swiglu_bwd": [P, P, P, I32, I32, P],
    "lsk_lora_down": [P, I64, P, P, I32, I32, F32, P, I32, P],
    "lsk_lora_du": [P, I64, I32, I32, P, I32, I32, P, I32, F32, P, P, I32, P],
    "lsk_lora_outer": [P, I64, I32, P, P, I32, I32, I32, I32, I32, P, I32, P, P],
    "lsk_lora_outer_noalloc": [P, I64, I32, P, P, I32, I32, I32, I32, I32, I32, P, P],
    "lsk_build_ext_fwd": [P, I32, I32, P, I32, I32, I32, I32, P, P],
    "lsk_build_ext_bwd": [P, P, I32, I32, P, P],
    "lsk_embed_gather": [P, P, P, I32, P, I32, I32, P],
    "lsk_vocab_logprob": [P, I32, I32, P, P, I32, P, P, P, P, P, P],
    "lsk_vocab_bwd": [P, I32, I32, P, P, I32, I32, P, P, P, P, P, I32, P],
    "lsk_wait_flag": [P, C.c_uint32, I64, P, P],
    "lsk_device_error": [C.POINTER(I32), I32],
}

_lib = None


def lib() -> C.CDLL:
    """The loaded libls.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libls.so not built ({LIB_PATH}); run python -m layer_streamed_nf4_dequant_b300.build")
        try:  # make the CUDA runtime torch uses visible first
            import torch  # noqa: F401
        except Exception:
            pass
        l = C.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            f = getattr(l, name)
            f.argtypes = args
            f.restype = C.c_int
        l.ls_last_error.argtypes = [P]
        l.ls_last_error.restype = C.c_char_p
        l.lsk_nf4_gemm_workspace_bytes.argtypes = []
        l.lsk_nf4_gemm_workspace_bytes.restype = U64
        _lib = l
    return _lib


def header_functions() -> list:
    """Function names declared in include/ls.h and include/ls_kernels.h."""
    names = []
    for h in HEADERS:
        txt = open(h).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s+([a-z_][a-z_0-9]*)\s*\(", txt, flags=re.M)
    return names


def last_error(ctx=None) -> str:
    m = lib().ls_last_error(ctx)
    return m.decode() if m else ""


def check(code: int, ctx=None) -> int:
    if code != 0:
        raise LSError(code, last_error(ctx))
    return code


def ptr(x) -> int | None:
    """Device/host address of a torch tensor (or pass through ints / None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def call(name: str, *args, ctx=None) -> int:
    f = getattr(lib(), name)
    conv = [ptr(a) if (a is None or hasattr(a, "data_ptr")) else a for a in args]
    return check(f(*conv), ctx)
