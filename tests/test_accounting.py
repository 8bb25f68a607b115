"""Work counts used by the benchmark, pinned to the counts the lesson prints."""
import json
import os

from exact_io_aware_08_gb300 import accounting as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_causal_tile_count_matches_page():
    g = json.load(open(os.path.join(GOLDEN, "causal_and_traffic_counts.json")))["causal_tiles"]
    assert W.causal_tiles(g["N"], g["B"]) == g["computed"]
    assert (g["N"] // g["B"]) ** 2 == g["total"]


def test_at_scale_counts_match_page():
    g = json.load(open(os.path.join(GOLDEN, "causal_and_traffic_counts.json")))["at_scale"]
    n, d = g["N"], g["d"]
    sig = lambda x: float(f"{x:.{g['printed_sig_figs']}g}")
    assert sig(W.fwd_flops(1, 1, n, n, d, False)) == g["fwd_flop_per_head"]
    assert sig(W.standard_traffic_elements(n, d)) == g["standard_traffic_elements_per_head"]
    assert sig(W.tiled_traffic_elements(n, d, g["Br"])) == g["flash_traffic_elements_per_head_no_cache"]
    assert g["heads"] * n * 4 == g["lse_bytes_all_heads"]


def test_pairs_and_flop_ratios():
    assert W.pairs(4, 4, True) == 10
    assert W.pairs(3, 5, False) == 15
    # the backward is 25% more matmul work than the four plain matmuls (10 vs 8 N^2 d)
    assert W.bwd_flops(1, 1, 64, 64, 32, False) * 8 == W.fwd_flops(1, 1, 64, 64, 32, False) * 20


def test_window_pairs_special_cases_and_brute_force():
    import numpy as np
    assert W.window_pairs(100, -1, 0) == W.pairs(100, 100, True)
    assert W.window_pairs(100, -1, -1) == W.pairs(100, 100, False)
    assert W.window_pairs(100, 0, 0) == 100
    for n, l, r in ((37, 5, 0), (37, 3, 9), (10, 20, 2), (64, -1, 7)):
        i = np.arange(n)[:, None]
        j = np.arange(n)[None, :]
        vis = np.ones((n, n), dtype=bool)
        if l >= 0:
            vis &= j >= i - l
        if r >= 0:
            vis &= j <= i + r
        assert W.window_pairs(n, l, r) == int(vis.sum())


def test_block_sparse_pairs_brute_force():
    import numpy as np
    g = np.random.default_rng(2)
    for n_q, n_kv, causal, block in ((37, 37, True, 4), (37, 29, False, 4), (300, 300, True, 128),
                                     (64, 64, False, 16)):
        nqb, nkb = -(-n_q // block), -(-n_kv // block)
        m = (g.random((2, 3, nqb, nkb)) < 0.5).astype(np.uint8)
        brute = 0
        for h in m.reshape(-1, nqb, nkb):
            i = np.arange(n_q)[:, None]
            j = np.arange(n_kv)[None, :]
            vis = h.astype(bool)[i // block, j // block]
            if causal:
                vis &= j <= i
            brute += int(vis.sum())
        assert W.block_sparse_pairs(m, n_q, n_kv, causal, block) == brute
    assert W.block_sparse_pairs(np.ones((3, 3)), 300, 300, True) == W.pairs(300, 300, True)
    assert W.block_sparse_pairs(np.ones((3, 3)), 300, 300, False) == W.pairs(300, 300, False)
