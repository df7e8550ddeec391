"""Host-side tile plan of the fused NF4 GEMM (lsk_nf4_gemm_plan; no GPU needed).

The plan is the host half of every NF4 product: tile shape, and whole tiles (one per
CTA) or the split schedule (one CTA per SM: round-robin whole tiles, then the remaining
tiles' k-iterations split evenly, partial tiles summed by the CTA that holds each
tile's first k-iteration).  These tests pin the cost model's choices on the Llama-3.1-8B
product shapes, and check the schedule invariants the device relies on by walking
each CTA's pieces as the kernel does (a restatement of its tile schedule): every
(tile, k-iteration) is computed exactly once, a share that starts inside a tile is
the only partial its CTA writes and is read by exactly one CTA, the one holding that
tile's first k-iteration, and every slot and flag index stays inside the scratch of
lsk_nf4_gemm_workspace_bytes().
"""
import random

import pytest

import layer_streamed_nf4_dequant_b300 as L

SMS = 148


def _pieces(c, p):
    """CTA c's pieces (tile, k0, k1): its round-robin whole tiles, then its share of the
    split k-iterations in (tile, k) order."""
    G, dp, I, ni = p["ctas"], p["whole_per_cta"], p["split_iters"], p["k_iters"]
    out = [(j * G + c, 0, ni) for j in range(dp)]
    pos, end = c * I // G, (c + 1) * I // G
    while pos < end:
        t, k0 = divmod(pos, ni)
        k1 = min(ni, k0 + (end - pos))
        out.append((dp * G + t, k0, k1))
        pos += k1 - k0
    return out


def _check_schedule(p):
    G, dp, I, ni = p["ctas"], p["whole_per_cta"], p["split_iters"], p["k_iters"]
    tiles = p["tiles_m"] * p["tiles_n"]
    if I == 0:
        assert G * dp == tiles or (dp == 1 and G == tiles)
        return
    assert 1 < G <= SMS and I >= G and I % ni == 0
    assert dp * G + I // ni == tiles
    owner = {}
    partial_of = {}
    for c in range(G):
        ps = _pieces(c, p)
        assert ps, "every CTA has work"
        for i, (t, k0, k1) in enumerate(ps):
            assert 0 <= t < tiles and 0 <= k0 < k1 <= ni
            for kk in range(k0, k1):
                assert (t, kk) not in owner
                owner[(t, kk)] = c
            if k0 > 0:
                assert i == dp and c not in partial_of   # only the first split piece
                partial_of[c] = t
    assert len(owner) == tiles * ni
    # the finisher of a split tile = owner of its k-iteration 0; its peers are the CTAs
    # whose shares start inside the tile, i.e. exactly the partials of that tile
    read_by = {}
    for c in range(G):
        for (t, k0, k1) in _pieces(c, p):
            if k0 == 0 and k1 < ni:
                tend = (t - dp * G + 1) * ni
                d = c + 1
                while d + 1 < G and (d + 1) * I // G < tend:
                    d += 1
                peers = list(range(c + 1, d + 1))
                assert peers == sorted(x for x, tt in partial_of.items() if tt == t)
                for x in peers:
                    assert x not in read_by
                    read_by[x] = c
    assert sorted(read_by) == sorted(partial_of)
    # scratch: one 256 x 256 fp32 slot and 8 epoch words per CTA
    ws = int(L.lib().lsk_nf4_gemm_workspace_bytes())
    assert 8192 + G * 256 * 256 * 4 <= ws and G * 8 * 4 <= 8192


# (mode, M, N, K) -> expected: whole tiles ("whole") or split with (whole rounds, split tiles)
PRODUCTS_8B = [
    ((0, 2048, 28672, 4096), (5, 156)),     # gate|up, shared-read forward rows
    ((0, 2048, 4096, 4096), "whole"),       # o: 128 tiles, one wave is cheaper than a split
    ((0, 2048, 6144, 4096), (0, 192)),      # q|k|v: 192 tiles = 1.3 waves
    ((0, 2048, 4096, 14336), (0, 128)),     # down: long reduction
    ((0, 1024, 28672, 4096), (2, 152)),     # recomputed policy forward
    ((0, 1024, 4096, 14336), (0, 64)),
    ((1, 1024, 28672, 4096), (0, 64)),      # input gradients: few output tiles
    ((1, 1024, 4096, 14336), (0, 224)),
    ((1, 1024, 6144, 4096), (0, 64)),
]


@pytest.mark.parametrize("spec,want", PRODUCTS_8B)
def test_plan_choices_on_8b_products(spec, want):
    p = L.gemm_plan(*spec)
    assert (p["nacc"], p["bn"]) == (2, 256)
    if want == "whole":
        assert p["split_iters"] == 0 and p["ctas"] == p["tiles_m"] * p["tiles_n"]
    else:
        rounds, split_tiles = want
        assert p["ctas"] == SMS and p["whole_per_cta"] == rounds
        assert p["split_iters"] == split_tiles * p["k_iters"]
    _check_schedule(p)


def test_plan_switches():
    spec = (0, 2048, 28672, 4096)
    # no scratch, or whole tiles asked for: never split
    for kw in ({"with_workspace": False}, {"split": -1}):
        p = L.gemm_plan(*spec, **kw)
        assert p["split_iters"] == 0 and p["ctas"] == p["tiles_m"] * p["tiles_n"]
    # 128 rows or fewer: no two-accumulator tile, no split, even when asked
    p = L.gemm_plan(0, 128, 4096, 4096, split=1)
    assert p["nacc"] == 1 and p["split_iters"] == 0
    # a forced one-accumulator tile cannot split
    p = L.gemm_plan(*spec, split=1, force_nacc=1)
    assert p["nacc"] == 1 and p["split_iters"] == 0
    # split asked for on a product the model would run whole
    p = L.gemm_plan(0, 2048, 4096, 4096, split=1)
    assert p["split_iters"] > 0
    _check_schedule(p)
    # 148 tiles: whole tiles, one per SM
    p = L.gemm_plan(0, 256, 148 * 256, 128, split=1)
    assert p["split_iters"] == 0 and p["ctas"] == 148 and p["whole_per_cta"] == 1
    # 296 tiles: two whole rounds on a persistent grid
    p = L.gemm_plan(0, 512, 148 * 256, 128, split=1)
    assert p["split_iters"] == 0 and p["ctas"] == 148 and p["whole_per_cta"] == 2
    # the LoRA stage is one more k-iteration per tile
    assert L.gemm_plan(0, 1024, 6144, 4096, ext_k=16)["k_iters"] == 65


def test_small_stack_products_take_small_whole_tiles():
    """The tiny test stack (hidden 256, 384 tokens): short reductions never split."""
    for spec in [(0, 384, 512, 256), (0, 384, 256, 512), (1, 384, 1024, 256), (1, 768, 512, 256)]:
        p = L.gemm_plan(*spec)
        assert p["split_iters"] == 0 and p["ctas"] == p["tiles_m"] * p["tiles_n"]


def test_split_schedule_invariants_random_shapes():
    rng = random.Random(7)
    for _ in range(150):
        mode = rng.randint(0, 1)
        M = rng.randint(129, 4096)
        N = 64 * rng.randint(1, 300)
        K = 64 * rng.randint(1, 120)
        ext = rng.choice([0, 0, 16, 32])
        p = L.gemm_plan(mode, M, N, K, ext_k=ext, split=1)
        if p["split_iters"] or p["whole_per_cta"] != 1:
            _check_schedule(p)
        out_cols = N if mode == 0 else K
        assert p["tiles_m"] == -(-M // (128 * p["nacc"])) and p["tiles_n"] == -(-out_cols // p["bn"])


def test_plan_rejects_bad_arguments():
    for args in [(2, 256, 256, 256), (0, 0, 256, 256), (0, 256, 100, 256), (0, 256, 256, 100)]:
        with pytest.raises(L.LSError):
            L.gemm_plan(*args)
    with pytest.raises(L.LSError):
        L.gemm_plan(0, 256, 256, 256, ext_k=8)
    with pytest.raises(L.LSError):
        L.gemm_plan(0, 256, 256, 256, split=2)


def test_paired_rows_plan():
    """Shared-read forward products (2T rows, pair_rows = T): a split plan pairs the
    halves (128-row blocks of one half, same counts as unpaired); a whole-tile plan, a
    one-accumulator tile or a batch that is not two halves falls back to whole tiles."""
    p = L.gemm_plan(0, 2048, 28672, 4096, pair_rows=1024)
    assert p["pair_rows"] == 1024 and (p["tiles_m"], p["tiles_n"]) == (8, 112)
    assert p["ctas"] == SMS and p["whole_per_cta"] == 5 and p["split_iters"] == 156 * 64
    _check_schedule(p)
    p = L.gemm_plan(0, 2048, 4096, 4096, pair_rows=1024)       # o: the model keeps whole tiles
    assert p["pair_rows"] == 0 and p["split_iters"] == 0 and p["ctas"] == p["tiles_m"] * p["tiles_n"]
    for kw in ({"pair_rows": 1000, "split": 1}, {"pair_rows": 1024, "split": 1, "force_nacc": 1}):
        p = L.gemm_plan(0, 2048, 28672, 4096, **kw)
        assert p["pair_rows"] == 0 and p["split_iters"] == 0 and p["ctas"] == p["tiles_m"] * p["tiles_n"]
    rng = random.Random(11)
    for _ in range(60):
        T = rng.randint(65, 2048)
        p = L.gemm_plan(rng.randint(0, 1), 2 * T, 64 * rng.randint(1, 200), 64 * rng.randint(1, 100),
                        split=1, pair_rows=T)
        assert p["pair_rows"] == T and p["tiles_m"] == -(-T // 128)
        if p["split_iters"] or p["whole_per_cta"] != 1:
            _check_schedule(p)
