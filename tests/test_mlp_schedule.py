"""The one-launch MLP's work decomposition, replayed on the CPU.

The persistent units of the swapped GEMM walk phase 0 (gate/up + SwiGLU:
whole tiles, the partial last wave split along K and, here, placed first)
and then phase 1 (down + residual: stream-K in groups of token tiles, a
range that crosses a weight tile's end taking the part after the crossing
first).  This mirror of the device-side scheduler (k_gemm_sab.cu, `Work`
with tail_first / defer, and the split choice of the launcher) checks, for
row counts from 1 to the largest the flags allow, that every gate/up tile
and every (token tile, weight tile, k-block) of the down projection is
covered exactly once, and that every down k-block reads a flag that some
gate/up tile's epilogue sets."""
import pytest

FM, BK = 128, 64


def work_items(p, num_kb, unit, n_units, cg, ext):
    n_ft = (p["n_ft"] + cg - 1) // cg
    items = []
    if p["stream_k"]:
        total = n_ft * num_kb
        groups = min(n_units // p["n_tt"], total)
        g, my_tt = unit // p["n_tt"], unit % p["n_tt"]
        w = total * g // groups if g < groups else 0
        w_end = total * (g + 1) // groups if g < groups else 0
        dw0 = dw1 = 0
        if ext and p["defer"] and w < w_end and w % num_kb:
            cross = (w // num_kb + 1) * num_kb
            if cross < w_end:
                dw0, dw1, w = w, cross, cross
        while True:
            if w >= w_end:
                if not ext or dw0 >= dw1:
                    break
                w, w_end, dw0 = dw0, dw1, dw1
            ft, kb0 = w // num_kb, w % num_kb
            kb1 = min(kb0 + (w_end - w), num_kb)
            w += kb1 - kb0
            items.append((my_tt, ft, kb0, kb1, -1))
        return items
    split, n_whole = p["split"], p["n_whole"]
    n_tail = p["n_tt"] * n_ft - n_whole if split > 1 else 0
    n_seg = n_tail * split
    tail_first = ext and p["tail_first"]
    w, w_end = unit, n_seg + n_whole
    while w < w_end:
        tile = w - n_seg + (n_tail if tail_first else 0)
        kb0, kb1, seg = 0, num_kb, -1
        if w < n_seg:
            tj, seg = w // split, w % split
            tile = tj if tail_first else n_whole + tj
            kb0, kb1 = num_kb * seg // split, num_kb * (seg + 1) // split
        items.append((tile % p["n_tt"], tile // p["n_tt"], kb0, kb1, seg))
        w += n_units
    return items


def launch_params(M, F, d, pairs):
    """The launcher's choices: token tiles, CTAs per MMA, units, tail split."""
    n_tt = (M + 255) // 256
    bt = ((M + n_tt - 1) // n_tt + 15) // 16 * 16
    cg = 2 if bt >= 32 else 1
    units = pairs if cg == 2 else 2 * pairs
    p0 = dict(n_tt=n_tt, n_ft=F // 64, stream_k=0, defer=0, tail_first=1)
    num_kb0 = (d + BK - 1) // BK
    tiles = n_tt * ((p0["n_ft"] + cg - 1) // cg)
    rem = tiles % units
    split = min(units // rem if rem else 1, num_kb0 // 8, 8)
    p0["split"], p0["n_whole"] = (split, tiles - rem) if split >= 2 else (1, tiles)
    p1 = dict(n_tt=n_tt, n_ft=(d + FM - 1) // FM, stream_k=1, defer=1, tail_first=0,
              split=1, n_whole=0)
    return p0, p1, cg, units


@pytest.mark.parametrize("M", [1, 9, 31, 32, 64, 89, 300, 524, 1000, 3136, 8192, 18688])
@pytest.mark.parametrize("F,d", [(14336, 4096), (12288, 4096)])
def test_every_tile_and_k_block_once_and_every_flag_set(M, F, d):
    p0, p1, cg, units = launch_params(M, F, d, pairs=76)
    assert (p0["n_ft"] + cg - 1) // cg * cg * p0["n_tt"] <= 16384 or M > 16384
    num_kb0, num_kb1 = (d + BK - 1) // BK, F // BK
    cover, flags = {}, set()
    for u in range(units):
        for tt, ft, kb0, kb1, seg in work_items(p0, num_kb0, u, units, cg, True):
            cover.setdefault((tt, ft), []).append((kb0, kb1))
            if seg <= 0:              # whole tile or the segment that finishes it
                flags.update((ft * cg + r, tt) for r in range(cg))
    n_pair_tiles = (p0["n_ft"] + cg - 1) // cg
    assert len(cover) == p0["n_tt"] * n_pair_tiles
    for segs in cover.values():
        segs.sort()
        assert segs[0][0] == 0 and segs[-1][1] == num_kb0
        assert all(a[1] == b[0] for a, b in zip(segs, segs[1:]))
    seen = set()
    for u in range(units):
        for tt, ft, kb0, kb1, _ in work_items(p1, num_kb1, u, units, cg, True):
            for kb in range(kb0, kb1):
                assert (tt, ft, kb) not in seen
                seen.add((tt, ft, kb))
                assert (kb, tt) in flags          # down k-block kb reads gate/up CTA tile kb
    assert len(seen) == p1["n_tt"] * ((p1["n_ft"] + cg - 1) // cg) * num_kb1


@pytest.mark.parametrize("M", [64, 524, 3136])
def test_the_extensions_reorder_the_work(M):
    """defer changes only the order of each unit's down-projection items;
    tail_first changes which tiles are split, not which tiles run."""
    p0, p1, cg, units = launch_params(M, 14336, 4096, pairs=76)
    for u in range(units):
        a = work_items(p1, 224, u, units, cg, True)
        b = work_items(p1, 224, u, units, cg, False)
        assert sorted(a) == sorted(b)
    tiles = lambda ext: sorted({i[:2] for u in range(units)
                                for i in work_items(p0, 64, u, units, cg, ext)})
    assert tiles(True) == tiles(False)
    if p0["split"] > 1:
        # the split tiles run first, so the last tiles to finish hold the
        # highest gate/up features
        firsts = [work_items(p0, 64, u, units, cg, True)[0] for u in range(units)]
        split_ft = {ft for _, ft, _, _, seg in firsts if seg >= 0}
        assert max(split_ft) < min(ft for u in range(units)
                                   for _, ft, _, _, seg in work_items(p0, 64, u, units, cg, True)
                                   if seg < 0) + 1


def test_the_library_rule_for_one_launch():
    """cb_debug_mlp_one_launch: one launch where both projections take the
    same swapped form and the flags fit, as the replay above assumes; the
    switches turn it off."""
    from rag_kv_cache_layer_gb300 import _lib as L
    one = lambda M, d=4096, F=14336: L.lib.cb_debug_mlp_one_launch(M, d, F)
    L.check(L.lib.cb_debug_mlp_fusion(1))
    L.check(L.lib.cb_debug_gemm_path(L.CB_GEMM_AUTO))
    for M in (1, 9, 64, 524, 3136, 8192, 18688):
        p0, _, cg, _ = launch_params(M, 14336, 4096, pairs=76)
        assert one(M) == 1, M
        assert (p0["n_ft"] + cg - 1) // cg * cg * p0["n_tt"] <= 16384
    assert one(18689) == 0 and one(66048) == 0       # the flags no longer fit
    assert one(12800, F=12288) == 1 and one(41472, F=12288) == 0
    assert one(0) == 0 and one(-5) == 0
    try:
        L.check(L.lib.cb_debug_mlp_fusion(0))
        assert one(524) == 0
        L.check(L.lib.cb_debug_mlp_fusion(1))
        L.check(L.lib.cb_debug_gemm_path(L.CB_GEMM_TOKEN_M))
        assert one(524) == 0                         # token rows on M: two launches
        L.check(L.lib.cb_debug_gemm_path(L.CB_GEMM_SWAP_AB))
        assert one(524) == 1
    finally:
        L.check(L.lib.cb_debug_mlp_fusion(1))
        L.check(L.lib.cb_debug_gemm_path(L.CB_GEMM_AUTO))
