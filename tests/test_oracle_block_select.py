"""Pins of the oracle's 128-token-block selection (CPU only).

- a hand-worked row (tests/golden/block_select_hand_example.txt);
- brute force in plain Python on tie-heavy rows: block maxima by loops, the
  order by a (score desc, block asc) sort, the emit page by page;
- when the table can hold every block, the result is the page-granular
  selection of every page.
"""
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_block_select_hand_example():
    lines = [l.split() for l in open(os.path.join(GOLD, "block_select_hand_example.txt"))
             if l.strip() and not l.startswith("#")]
    sc = np.zeros((1, 40), np.float32)
    sc[0, 38:] = -np.inf
    sc[0, [3, 9, 20, 33]] = [5.0, 2.0, 5.0, -1.0]
    bt = np.array([[10, 11, 12, 13, 14]], np.int32)
    for i in range(0, len(lines), 3):
        ft = lines[i][0] == "1"
        ti_e = [int(x) for x in lines[i][1:]]
        sb_e = [int(x) for x in lines[i + 1][1:]]
        ctx_e = int(lines[i + 2][1])
        ti, sb, ctx = O.topk_select_blocks(sc, np.zeros(1, np.int32), np.array([600], np.int32), bt, 0, 24, ft)
        m = len(ti_e)
        assert ti[0, :m].tolist() == ti_e and (ti[0, m:] == -1).all()
        assert sb[0, :m].tolist() == sb_e and (sb[0, m:] == -1).all()
        assert ctx[0] == ctx_e


def brute(scores, L, bt_row, id_rule, k_pages, force_tail, max_pages):
    L = max(0, min(int(L), max_pages * 16))
    n = (L + 15) // 16
    nb = (n + 7) // 8
    kb = min(k_pages // 8, nb)
    ti = [-1] * k_pages
    sb = [-1] * k_pages
    if kb == 0:
        return ti, sb, 0
    bscore = []
    for b in range(nb):
        best = None
        for p in range(8 * b, min(8 * b + 8, n)):
            v = float(scores[p])
            best = v if best is None or v > best else best
        bscore.append(best)
    cands = list(range(nb - 1 if force_tail else nb))
    cands.sort(key=lambda b: (-bscore[b], b))
    take = cands[:kb - 1 if force_tail else kb]
    if force_tail:
        take.append(nb - 1)
    take.sort()
    m, ctx = 0, 0
    for b in take:
        for p in range(8 * b, min(8 * b + 8, n)):
            ti[m] = p
            blk = int(bt_row[b])
            sb[m] = blk * 16 + p % 8 if id_rule == 0 else blk * 8 + p % 8
            ctx += L - 16 * (n - 1) if p == n - 1 else 16
            m += 1
    return ti, sb, ctx


@pytest.mark.parametrize("id_rule", [0, 1])
@pytest.mark.parametrize("force_tail", [True, False])
def test_block_select_brute_force(id_rule, force_tail):
    rng = np.random.default_rng(11 + id_rule + 2 * force_tail)
    max_pages = 96
    lens = [0, 1, 15, 16, 17, 127, 128, 129, 255, 256, 300, 777, 1000, 1536, 1537, 96 * 16, 5000, -3]
    rows = len(lens) * 4
    row_len = np.array(lens * 4, np.int32)
    # scores from a small set of values: many equal block maxima
    sc = rng.integers(-3, 4, size=(rows, max_pages)).astype(np.float32) * 0.5
    bt = rng.permutation(rows * 12).astype(np.int32).reshape(rows, 12)
    rs = np.arange(rows, dtype=np.int32)
    for k_pages in (8, 16, 23, 40, 128):
        ti, sb, ctx = O.topk_select_blocks(sc, rs, row_len, bt, id_rule, k_pages, force_tail)
        for r in range(rows):
            e_ti, e_sb, e_ctx = brute(sc[r], row_len[r], bt[r], id_rule, k_pages, force_tail, max_pages)
            assert ti[r].tolist() == e_ti, (k_pages, r)
            assert sb[r].tolist() == e_sb, (k_pages, r)
            assert ctx[r] == e_ctx, (k_pages, r)


def test_every_block_is_every_page():
    rng = np.random.default_rng(3)
    rows, max_pages = 12, 64
    sc = rng.standard_normal((rows, max_pages)).astype(np.float32)
    row_len = np.array([1, 16, 100, 128, 129, 500, 640, 1000, 1023, 1024, 17, 300], np.int32)
    bt = rng.permutation(rows * 8).astype(np.int32).reshape(rows, 8)
    rs = np.arange(rows, dtype=np.int32)
    for id_rule in (0, 1):
        a = O.topk_select_blocks(sc, rs, row_len, bt, id_rule, 64, True)
        b = O.topk_select(sc, rs, row_len, bt, id_rule, 64, True)
        for x, y in zip(a, b):
            assert np.array_equal(x, y)
