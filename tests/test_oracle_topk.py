"""Pins of the oracle's kept-token selection: hand-worked golden cases, an exhaustive
search over all candidate subsets on tiny inputs (the kept set is the unique subset whose
every member beats every dropped candidate under score-descending, position-ascending
order), and the selection invariants on larger random inputs."""
import itertools
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "topk_small.json")


def test_golden_hand_worked_cases():
    cases = json.load(open(GOLDEN))["cases"]
    assert len(cases) >= 5
    for c in cases:
        L = c["len"]
        scores = np.zeros((1, 1, L), dtype=np.float32)
        scores[0, 0, :] = c["scores"]
        kept, kl = oracle.select_topk(scores, np.array([L], dtype=np.int32), c["n_sink"],
                                      c["n_recent"], c["k_top"])
        assert kl[0] == len(c["kept"]), c
        assert kept[0, 0, :kl[0]].tolist() == c["kept"], c


def _beats(sa, pa, sb, pb):
    return sa > sb or (sa == sb and pa < pb)


@pytest.mark.parametrize("seed", range(12))
def test_exhaustive_subset_search(seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(8, 14))
    n_sink, n_recent = int(rng.integers(0, 3)), int(rng.integers(0, 3))
    k_top = int(rng.integers(1, 5))
    if n_sink + n_recent + k_top >= L:
        k_top = max(1, L - n_sink - n_recent - 2)
    pool = np.array([0.0, -0.0, 1.0, 2.0, -1.5, 0.25], dtype=np.float32)   # many ties
    s = pool[rng.integers(0, len(pool), size=(2, L))]
    scores = s.reshape(1, 2, L).astype(np.float32)
    kept, kl = oracle.select_topk(scores, np.array([L], dtype=np.int32), n_sink, n_recent, k_top)
    cand = list(range(n_sink, L - n_recent))
    for g in range(2):
        valid = []
        for sub in itertools.combinations(cand, k_top):
            rest = [c for c in cand if c not in sub]
            if all(_beats(s[g, a], a, s[g, b], b) for a in sub for b in rest):
                valid.append(sub)
        assert len(valid) == 1
        expect = sorted(set(range(n_sink)) | set(valid[0]) | set(range(L - n_recent, L)))
        assert kept[0, g, :kl[0]].tolist() == expect


def test_invariants_large_random():
    rng = np.random.default_rng(7)
    B, H, S = 3, 4, 5000
    lens = np.array([5000, 400, 2345], dtype=np.int32)
    scores = rng.exponential(size=(B, H, S)).astype(np.float32)
    scores[0, 0, 100:200] = 3.25                     # a block of ties straddling the cut
    n_sink, n_recent, k_top = 4, 256, 64
    kept, kl = oracle.select_topk(scores, lens, n_sink, n_recent, k_top)
    K = n_sink + n_recent + k_top
    for b in range(B):
        L = int(lens[b])
        assert kl[b] == min(L, K)
        for g in range(H):
            row = kept[b, g, :kl[b]]
            assert np.all(np.diff(row) > 0)
            if L <= K:
                assert row.tolist() == list(range(L))
                continue
            assert set(range(n_sink)) <= set(row.tolist())
            assert set(range(L - n_recent, L)) <= set(row.tolist())
            cands = [t for t in row.tolist() if n_sink <= t < L - n_recent]
            assert len(cands) == k_top
            dropped = sorted(set(range(n_sink, L - n_recent)) - set(cands))
            ks, ds = scores[b, g, cands], scores[b, g, dropped]
            assert ks.min() >= ds.max()
            thr = ks.min()
            if np.any(ds == thr):                   # ties at the cut: kept positions are lower
                assert max(c for c in cands if scores[b, g, c] == thr) < \
                    min(d for d in dropped if scores[b, g, d] == thr)


def test_nan_is_refused():
    scores = np.ones((1, 1, 40), dtype=np.float32)
    scores[0, 0, 10] = np.nan
    with pytest.raises(oracle.OracleError):
        oracle.select_topk(scores, np.array([40], dtype=np.int32), 2, 4, 5)
