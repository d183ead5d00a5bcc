"""Host logic of bench.py: the visible-pair count behind the FLOPs of the
mask variants, against a brute-force count of the mask definition (query i
sees key j iff lo_i <= j < hi_i, cudnn-frontend PR #554 `sdpa` masks)."""
import itertools

import bench


def _brute(s_q, s_kv, mask, window):
    delta = s_kv - s_q if mask == 2 else 0
    n = 0
    for i, j in itertools.product(range(s_q), range(s_kv)):
        if mask != 0 and j > i + delta:
            continue
        if window >= 0 and j < i + delta - window:
            continue
        n += 1
    return n


def test_visible_pairs_matches_brute_force():
    for s_q, s_kv in [(1, 1), (7, 7), (5, 13), (13, 5), (32, 32)]:
        for mask in (0, 1, 2):
            for window in (-1, 0, 3, 40):
                assert bench.visible_pairs(s_q, s_kv, mask, window) == _brute(s_q, s_kv, mask,
                                                                               window)


def test_visible_pairs_closed_forms():
    s, w = 16384, 2048
    assert bench.visible_pairs(s, s, 1, -1) == s * (s + 1) // 2
    assert bench.visible_pairs(s, s, 1, w) == w * (w + 1) // 2 + (s - w) * (w + 1)
    assert bench.visible_pairs(4096, s, 2, -1) == 4096 * (s - 4096) + 4096 * 4097 // 2
    assert bench.visible_pairs(300, 500, 0, -1) == 300 * 500
