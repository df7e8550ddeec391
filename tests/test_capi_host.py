"""Host-side checks of the C ABI (no GPU): exports, quantiser, planner, layout."""
import ctypes as C
import math

import numpy as np
import pytest

import layer_streamed_nf4_dequant_b300 as L
import oracle
import synth


def test_library_exports_every_header_function():
    lib = L.lib()
    names = L.header_functions()
    assert len(names) >= 30
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


@pytest.mark.parametrize("shape", [(3, 64), (17, 256), (64, 896)])
def test_host_quantizer_bit_exact_vs_oracle(shape):
    rng = np.random.default_rng(shape[1])
    w = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    w[0, :64] = 0.0                                  # zero block
    w[-1, -64:] = np.tile(oracle.NF4_TABLE, 4) * 3   # exact code points
    mids = ((oracle.NF4_TABLE[:-1].astype(np.float64) + oracle.NF4_TABLE[1:]) / 2).astype(np.float32)
    if shape[0] > 1:
        w[1, :15] = mids
        w[1, 15] = 1.0
    pk, am = L.quantize_host(w)
    codes, absmax = oracle.nf4_quantize(w)
    np.testing.assert_array_equal(am, absmax)
    np.testing.assert_array_equal(pk, oracle.nf4_pack(codes))


def test_host_quantizer_large_matrix_threads():
    w = synth.weight(synth.LAYER_896, 0, "gate")    # 4864 x 896
    pk1, am1 = L.quantize_host(w, nthreads=1)
    pk8, am8 = L.quantize_host(w, nthreads=8)
    np.testing.assert_array_equal(pk1, pk8)
    np.testing.assert_array_equal(am1, am8)
    codes, absmax = oracle.nf4_quantize(w[:512])
    np.testing.assert_array_equal(pk1[:512], oracle.nf4_pack(codes))


def test_quantizer_rejects_bad_shape():
    w = np.zeros((2, 65), np.float32)
    rc = L.lib().nf4_quantize(w.ctypes.data, 2, 65, w.ctypes.data, w.ctypes.data, 1)
    assert rc == L.LS_ERR_ARG


def test_plan_and_preflight_refusal():
    s32 = synth.QWEN_32B
    cfg = L.make_config(s32)
    need = L.plan_bytes(cfg)                     # fits the 4 GiB cap of the 32B workload
    assert 0 < need <= s32.cap_bytes
    small = L.make_config(s32, cap_bytes=1 << 30)
    n = C.c_uint64(0)
    rc = L.lib().ls_plan(C.byref(small), C.byref(n))
    assert rc == L.LS_ERR_CAP and n.value == need
    assert "exceeds the cap" in L.last_error()
    bad = L.make_config(synth.LLAMA_8B)
    bad.head_dim = 96
    assert L.lib().ls_plan(C.byref(bad), C.byref(n)) == L.LS_ERR_ARG


def test_layer_layout_sizes():
    s = synth.LLAMA_8B
    offs, nbytes = L.layer_layout(L.make_config(s))
    H, I, nq, nkv = s.hidden, s.inter, s.heads * s.head_dim, s.kv_heads * s.head_dim
    params = (nq + 2 * nkv) * H + H * nq + 2 * I * H + H * I
    # packed 0.5 B + absmax 4/64 B per weight, two bf16 norms, 256-byte alignment slack
    assert abs(nbytes - (params * 0.5625 + 4 * H)) < 16 * 256
    assert offs == sorted(offs) and offs[0] == 0
    assert offs[1] - offs[0] == nq * H // 2 and offs[2] - offs[1] == nkv * H // 2
    assert offs[5] - offs[4] == I * H // 2
    assert nbytes / 1e6 == pytest.approx(122.7, abs=0.1)


def test_rope_table_matches_fp64():
    maxp, hd, theta = 300, 128, 5e5
    c = np.empty((maxp, hd // 2), np.float32)
    s = np.empty_like(c)
    L.check(L.lib().ls_rope_table(c.ctypes.data, s.ctypes.data, maxp, hd, theta))
    ang = np.arange(maxp)[:, None] * theta ** (-2.0 * np.arange(hd // 2) / hd)[None, :]
    np.testing.assert_array_equal(c, np.cos(ang).astype(np.float32))
    np.testing.assert_array_equal(s, np.sin(ang).astype(np.float32))


def test_gemm_split_workspace_size():
    """Epoch words (8 KiB) plus one 256 x 256 fp32 partial tile for each of 148 CTAs."""
    assert int(L.lib().lsk_nf4_gemm_workspace_bytes()) == 8192 + 148 * 256 * 256 * 4


def test_binding_signatures_match_header_declarations():
    """Every function declared in include/*.h has a ctypes signature with the same number
    of parameters (catches ABI drift between the headers and the binding)."""
    import re
    from layer_streamed_nf4_dequant_b300 import _binding as B
    decl = {}
    for h in B.HEADERS:
        txt = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s+([a-z_][a-z_0-9]*)\s*\(([^)]*)\)\s*;", txt,
                             flags=re.M):
            args = m.group(2).strip()
            decl[m.group(1)] = 0 if args in ("", "void") else len(args.split(","))
    assert sorted(decl) == sorted(L.header_functions())
    special = {"ls_last_error": 1, "lsk_nf4_gemm_workspace_bytes": 0}
    lib = L.lib()
    for name, n in decl.items():
        if name in special:
            assert n == special[name] and len(getattr(lib, name).argtypes) == n, name
        else:
            assert name in B._SIGS, f"{name} has no ctypes signature"
            assert len(B._SIGS[name]) == n, f"{name}: header {n} parameters, binding {len(B._SIGS[name])}"


def test_attention_and_wait_entry_points_refuse_bad_arguments_on_the_host():
    """Argument checks that run before anything touches the device (so no GPU is needed):
    the tensor-core attention kernels need 16-byte aligned operands (TMA, 16-byte
    stores), a head dimension of 64 or 128, a whole number of query heads per
    key/value head, row pitches that hold a whole row and a grid within CUDA's limits; the
    bounded wait needs a 4-byte aligned flag and a limit >= 0."""
    lib = L.lib()
    A, B, C_, D = 0x10000, 0x20000, 0x30000, 0x40000       # 16-byte aligned stand-ins
    # forward: qkv not 16-byte aligned; head_dim 96; 5 query heads on 2 kv heads
    assert lib.lsk_attn_fwd(A + 8, 768, B, 1, 64, 4, 1, 128, C_, 512, D, 64, None) == L.LS_ERR_ARG
    assert lib.lsk_attn_fwd(A, 768, B, 1, 64, 4, 1, 96, C_, 512, D, 64, None) == L.LS_ERR_ARG
    assert lib.lsk_attn_fwd(A, 1152, B, 1, 64, 5, 2, 128, C_, 640, D, 64, None) == L.LS_ERR_ARG
    assert "lsk_attn_fwd" in L.last_error()
    # backward: no kv heads; dqkv row pitch not a multiple of 4; head-split scratch misaligned
    args = [A, 768, B, C_, 512, D, B, 1, 64, 4, 1, 128, C_, D, 768, 64]
    bad_kv = list(args)
    bad_kv[10] = 0
    assert lib.lsk_attn_bwd(*bad_kv, None, None) == L.LS_ERR_ARG
    bad_ldg = list(args)
    bad_ldg[14] = 770
    assert lib.lsk_attn_bwd(*bad_ldg, None, None) == L.LS_ERR_ARG
    assert lib.lsk_attn_bwd(*args, D + 4, None) == L.LS_ERR_ARG
    # ... forward output misaligned (8-byte reads of it); row pitches narrower than a row
    bad_o = list(args)
    bad_o[3] = C_ + 4
    assert lib.lsk_attn_bwd(*bad_o, None, None) == L.LS_ERR_ARG
    for i, v in ((1, 760), (4, 504), (14, 764)):      # ld, lddo, ldg one step short
        narrow = list(args)
        narrow[i] = v
        assert lib.lsk_attn_bwd(*narrow, None, None) == L.LS_ERR_ARG
    # ... grid limits: 65536 sequences; 65536 query tiles
    many = list(args)
    many[7] = 65536
    assert lib.lsk_attn_bwd(*many, None, None) == L.LS_ERR_ARG
    long_ = list(args)
    long_[8] = 65536 * 128 + 1
    assert lib.lsk_attn_bwd(*long_, None, None) == L.LS_ERR_ARG
    assert "lsk_attn_bwd" in L.last_error()
    # forward: output pitch narrower than nh * head_dim; grid limits
    assert lib.lsk_attn_fwd(A, 768, B, 1, 64, 4, 1, 128, C_, 504, D, 64, None) == L.LS_ERR_ARG
    assert lib.lsk_attn_fwd(A, 768, B, 65536, 64, 4, 1, 128, C_, 512, D, 64, None) == L.LS_ERR_ARG
    assert lib.lsk_attn_fwd(A, 768, B, 1, 65536 * 128 + 1, 4, 1, 128, C_, 512, D, 64, None) == L.LS_ERR_ARG
    # bounded wait: misaligned flag; negative limit; no status
    assert lib.lsk_wait_flag(A + 2, 0, 1000, B, None) == L.LS_ERR_ARG
    assert lib.lsk_wait_flag(A, 0, -1, B, None) == L.LS_ERR_ARG
    assert lib.lsk_wait_flag(A, 0, 1000, None, None) == L.LS_ERR_ARG


def test_kernel_entry_points_refuse_misaligned_pointers_on_the_host():
    """The kernels move whole 4-, 8- and 16-byte words, so a pointer below a call's
    alignment would fault on the device: each call refuses it with LS_ERR_ARG before
    any launch (no GPU needed).  Each case shifts one pointer of an otherwise valid call."""
    lib = L.lib()
    A, B, C_, D, E, F = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000   # 16-byte aligned
    ws = 0x100000
    wsb = int(lib.lsk_nf4_gemm_workspace_bytes())
    cases = [
        # dequant: codes 4-byte, output 16-byte
        ("lsk_nf4_dequant", [A + 2, B, 4, 64, C_, None]),
        ("lsk_nf4_dequant", [A, B, 4, 64, C_ + 8, None]),
        # GEMM: activation, codes, output, residual 16-byte; absmax 4-byte
        ("lsk_nf4_gemm", [0, A + 8, 64, 16, B, C_, 64, 64, None, None, 0, 0, D, 64, None, 0, 0, 0, None]),
        ("lsk_nf4_gemm", [0, A, 64, 16, B + 8, C_, 64, 64, None, None, 0, 0, D, 64, None, 0, 0, 0, None]),
        ("lsk_nf4_gemm", [0, A, 64, 16, B, C_ + 2, 64, 64, None, None, 0, 0, D, 64, None, 0, 0, 0, None]),
        ("lsk_nf4_gemm", [0, A, 64, 16, B, C_, 64, 64, None, None, 0, 0, D + 8, 64, None, 0, 0, 0, None]),
        ("lsk_nf4_gemm", [0, A, 64, 16, B, C_, 64, 64, None, None, 0, 0, D, 64, E + 8, 64, 0, 0, None]),
        ("lsk_nf4_gemm", [0, A, 64, 16, B, C_, 64, 64, E + 8, F, 16, 0, D, 64, None, 0, 0, 0, None]),
        ("lsk_nf4_gemm_sk", [1, A, 64, 16, B, C_, 64, 64, None, None, 0, 1, D + 4, 64, None, 0, 0, 0, 0, 0,
                             ws, wsb, None]),
        # RMSNorm: forward 16-byte; backward fp32 16-byte, bf16 8-byte
        ("lsk_rmsnorm_fwd", [A + 8, B, C_, D, 4, 64, 1e-5, None]),
        ("lsk_rmsnorm_bwd", [A + 8, B, C_, D, E, None, 4, 64, 0, None]),
        ("lsk_rmsnorm_bwd", [A, B + 4, C_, D, E, None, 4, 64, 0, None]),
        ("lsk_rmsnorm_bwd", [A, B, C_, D, E, F + 4, 4, 64, 0, None]),
        # SwiGLU: forward 16-byte; backward dh 16-byte, bf16 8-byte
        ("lsk_swiglu_fwd", [A + 8, B, 4, 64, None]),
        ("lsk_swiglu_bwd", [A, B + 4, C_, 4, 64, None]),
        # LoRA: projections read 4-byte words; the outer product writes float2 partials
        ("lsk_lora_down", [A + 2, 64, B, C_, 16, 64, 1.0, D, 4, None]),
        ("lsk_lora_down", [A, 64, B + 2, C_, 16, 64, 1.0, D, 4, None]),
        ("lsk_lora_du", [A + 2, 64, 0, 16, B, 16, 16, C_, 16, 1.0, D, E, 4, None]),
        ("lsk_lora_outer", [A, 64, 64, B, None, 16, 16, 4, 0, 0, C_ + 4, 4, D, None]),
        # embedding rows 16-byte, codes 4-byte; vocabulary products as the GEMM
        ("lsk_embed_gather", [A, B + 2, C_, 128, D, 4, 64, None]),
        ("lsk_embed_gather", [A, B, C_, 128, D + 8, 4, 64, None]),
        ("lsk_vocab_logprob", [A + 8, 4, 64, B, C_, 128, D, E, F, F, F, None]),
        ("lsk_vocab_bwd", [A, 4, 64, B, C_, 0, 64, D, E, F, F, A + 0x1000 + 8, 0, None]),
        ("lsk_vocab_bwd", [A, 4, 64, B, C_, 0, 64, D, E, F, A + 0x1000, A + 0x2000 + 4, 0, None]),
    ]
    for name, args in cases:
        assert getattr(lib, name)(*args) == L.LS_ERR_ARG, (name, args)
        assert name in L.last_error()
    # build_ext: row counts whose element count overflows int32
    assert lib.lsk_build_ext_fwd(A, 0, 16, None, 0, 0, 16, 2 ** 31 // 64 + 1, B, None) == L.LS_ERR_ARG
    assert lib.lsk_build_ext_bwd(A, None, 16, 2 ** 31 // 64 + 1, B, None) == L.LS_ERR_ARG
