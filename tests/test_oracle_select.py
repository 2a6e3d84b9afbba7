"""Pins of the oracle's two-level selection ("DeepSeek-V4.1-Flash-NVFP4" §3.3:
blocks of 8 positions scored by their best position, top-2048 blocks with the
block holding the newest position always kept, then top-512 positions; config
walkthrough §2.1 for the sizes). Ties go to the lower index (the pages are silent
on ties; the lower index is the reading taken). Checked by brute force on tiny
inputs with many ties."""
import itertools

import numpy as np

from oracle import oracle as orc


def brute_select(scores, blk, Kb, Kp):
    n = len(scores)
    if n == 0:
        return []
    nb = -(-n // blk)
    bm = [max(scores[b * blk:(b + 1) * blk]) for b in range(nb)]
    if nb <= Kb:
        kept = set(range(nb))
    else:
        newest = (n - 1) // blk
        others = sorted((b for b in range(nb) if b != newest), key=lambda b: (-bm[b], b))
        kept = set(others[:Kb - 1]) | {newest}
    cand = [t for t in range(n) if t // blk in kept]
    best = sorted(cand, key=lambda t: (-scores[t], t))[:Kp]
    return sorted(best)


def test_matches_brute_force_with_ties():
    rng = np.random.default_rng(0)
    for trial in range(400):
        n = int(rng.integers(0, 70))
        levels = rng.integers(1, 6)
        s = rng.integers(0, levels, n).astype(np.float32) * np.float32(0.5)
        blk, Kb, Kp = 8, int(rng.integers(1, 5)), int(rng.integers(1, 12))
        idx, m = orc.select(s, blk, Kb, Kp)
        ref = brute_select(list(s), blk, Kb, Kp)
        assert m == len(ref)
        assert list(idx[:m]) == ref and np.all(idx[m:] == -1), (trial, n, Kb, Kp)


def test_exhaustive_tiny():
    for n in range(1, 11):
        for s in itertools.product([0.0, 1.0], repeat=min(n, 6)):
            s = np.array(list(s) + [0.5] * (n - len(s)), np.float32)
            idx, m = orc.select(s, 2, 2, 3)
            assert list(idx[:m]) == brute_select(list(s), 2, 2, 3)


def test_newest_block_always_kept_even_when_worst():
    s = np.ones(8 * 40, np.float32)
    s[-8:] = -5.0  # the newest block has the lowest scores
    idx, m = orc.select(s, 8, 4, 32)
    kept_blocks = set(int(t) // 8 for t in idx[:m])
    assert 39 in kept_blocks and len(kept_blocks) == 4
    assert m == 32  # 4 blocks x 8 positions, all kept


def test_block_stage_is_identity_when_few_blocks():
    rng = np.random.default_rng(1)
    s = rng.standard_normal(2048).astype(np.float32)  # 256 blocks <= 2048
    idx, m = orc.select(s, 8, 2048, 512)
    ref = np.sort(np.argsort(-s, kind="stable")[:512])
    assert m == 512 and np.array_equal(idx, ref)


def test_short_context_keeps_everything():
    s = np.arange(100, dtype=np.float32)
    idx, m = orc.select(s, 8, 2048, 512)
    assert m == 100 and np.array_equal(idx[:100], np.arange(100)) and np.all(idx[100:] == -1)
    idx, m = orc.select(np.zeros(0, np.float32), 8, 2048, 512)
    assert m == 0 and np.all(idx == -1)


def test_planted_high_scores_are_selected_and_the_block_cut_binds():
    rng = np.random.default_rng(2)
    n = 8 * 5000
    s = rng.standard_normal(n).astype(np.float32)
    plants = rng.choice(n - 8, 16, replace=False)
    s[plants] = 100.0
    idx, m = orc.select(s, 8, 2048, 512)
    assert m == 512 and set(plants) <= set(idx.tolist())
    assert len(set(int(t) // 8 for t in idx)) <= 2048


def flat_top(scores, Kp):
    """The Kp best positions by (score desc, position asc), ascending."""
    order = np.lexsort((np.arange(len(scores)), -scores.astype(np.float64)))
    return np.sort(order[:Kp])


def top_within_top_blocks(scores, blk, Kp):
    """The Kp best positions among the positions of the Kp best blocks (blocks by
    (block max desc, block asc)), ascending."""
    n = len(scores)
    nb = -(-n // blk)
    bm = np.array([scores[b * blk:(b + 1) * blk].max() for b in range(nb)], np.float64)
    blocks = np.lexsort((np.arange(nb), -bm))[:Kp]
    cand = np.concatenate([np.arange(b * blk, min(n, b * blk + blk)) for b in np.sort(blocks)])
    order = np.lexsort((cand, -scores[cand].astype(np.float64)))
    return np.sort(cand[order[:Kp]])


def test_two_levels_equal_the_flat_top_when_blocks_outnumber_positions():
    # With the block score the maximum of its positions' scores and more blocks kept
    # than positions (Kb - 1 >= Kp; the pages' 2047 >= 512), the two-level rule returns
    # the Kp best positions overall, and those lie among the positions of the Kp best
    # blocks: a best position's block ranks at least as high as that position, and
    # the blocks of the Kp best positions form a top set of the block order, so the
    # Kb - 1 best blocks other than the newest already contain them. The newest
    # block, kept regardless, changes nothing then. (With Kb = Kp it can: the
    # brute-force test above covers that regime.)
    rng = np.random.default_rng(3)
    for trial in range(300):
        n = int(rng.integers(1, 200))
        blk = int(rng.integers(1, 5))
        Kp = int(rng.integers(1, 12))
        Kb = Kp + 1 + int(rng.integers(0, 6))
        s = rng.integers(0, int(rng.integers(1, 7)), n).astype(np.float32)
        if trial % 3 == 0:
            s[(n - 1) // blk * blk:] = -9.0  # the newest block is the worst
        idx, m = orc.select(s, blk, Kb, Kp)
        ref = flat_top(s, Kp)
        assert m == len(ref) and np.array_equal(idx[:m], ref), (trial, n, blk, Kb, Kp)
        assert np.array_equal(top_within_top_blocks(s, blk, Kp), ref), trial


def test_two_levels_equal_the_flat_top_at_the_pages_sizes():
    rng = np.random.default_rng(4)
    for n in (16385, 20011, 65536):  # 2,049 to 8,192 blocks of 8
        for levels in (3, 50, 0):
            s = (rng.integers(0, levels, n).astype(np.float32) if levels
                 else rng.standard_normal(n).astype(np.float32))
            s[(n - 1) // 8 * 8:] = -100.0  # newest block last
            idx, m = orc.select(s, 8, 2048, 512)
            ref = flat_top(s, 512)
            assert m == 512 and np.array_equal(idx, ref), (n, levels)
            assert np.array_equal(top_within_top_blocks(s, 8, 512), ref), (n, levels)


def top_above_threshold(scores, blk, Kp, t):
    """The Kp best positions by (score desc, position asc), ascending, among the
    positions at or above t of the blocks whose maximum is at or above t."""
    n = len(scores)
    nb = -(-n // blk)
    bm = np.array([scores[b * blk:(b + 1) * blk].max() for b in range(nb)], np.float64)
    blocks = np.nonzero(bm >= t)[0]
    cand = np.concatenate([np.arange(b * blk, min(n, b * blk + blk)) for b in blocks])
    cand = cand[scores[cand] >= t]
    order = np.lexsort((cand, -scores[cand].astype(np.float64)))
    return np.sort(cand[order[:Kp]])


def test_any_threshold_that_kp_blocks_reach_keeps_the_answer():
    # The selection kernel's candidates: for any t that at least Kp block maxima
    # reach, the Kp best positions all score at least t (each of the Kp best blocks
    # holds a position at or above the Kp-th best block maximum, which is at least
    # t), so they lie among the positions at or above t of the blocks whose maximum
    # reaches t, and the Kp best of those are the rule's answer. Thresholds from the
    # largest one (the Kp-th best block maximum) down to below every score, with
    # ties, partial newest blocks and Kb - 1 >= Kp.
    rng = np.random.default_rng(9)
    for trial in range(400):
        blk = int(rng.integers(1, 9))
        Kp = int(rng.integers(1, 40))
        Kb = Kp + 1 + int(rng.integers(0, 8))
        n = int(rng.integers(1, 600))
        levels = int(rng.integers(0, 8))
        s = (rng.integers(0, levels, n).astype(np.float32) if levels
             else rng.standard_normal(n).astype(np.float32))
        idx, m = orc.select(s, blk, Kb, Kp)
        nb = -(-n // blk)
        bm = np.sort(np.array([s[b * blk:(b + 1) * blk].max() for b in range(nb)], np.float64))[::-1]
        if nb < Kp:
            continue  # every block is a candidate: nothing to choose
        t_max = bm[Kp - 1]
        for t in (t_max, t_max - 0.5, bm[-1], bm[-1] - 1.0, float(rng.uniform(bm[-1] - 1.0, t_max))):
            assert (bm >= t).sum() >= Kp
            got = top_above_threshold(s, blk, Kp, t)
            assert len(got) == m and np.array_equal(got, idx[:m]), (trial, n, blk, Kp, t)


def test_a_threshold_above_the_kp_th_block_maximum_can_lose_positions():
    # The bound is tight: above the Kp-th best block maximum fewer than Kp blocks
    # remain and the answer is not kept (the kernel never uses such a threshold).
    s = np.array([5, 0, 0, 0, 4, 0, 0, 0, 3, 0, 0, 0], np.float32)
    idx, m = orc.select(s, 4, 3, 2)
    assert list(idx[:m]) == [0, 4]
    assert list(top_above_threshold(s, 4, 2, 4.5)) == [0]
