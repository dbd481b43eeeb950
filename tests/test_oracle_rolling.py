"""Pins of the oracle's rolling admission (oracle.rolling_admit) to facts outside it.

  * static-score invariant: when every token's score is fixed, admitting the tokens one step at
    a time keeps exactly the set a fresh selection over the whole sequence keeps (each token
    leaving the recent window meets the current top-k set once, and the top-k of the tokens
    seen so far is what survives) -- checked against the oracle's top-k selection;
  * data integrity: every slot holds the K/V rows of the position it records;
  * hand-built ties: equal lowest scores drop the highest position; a leaving token whose
    score equals the lowest is the one dropped; k_top = 0 keeps sinks and the recent window;
  * refusals: NaN scores, a state whose leaving token is missing.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import bits, rand_bf16


def _pool(B, hkv, cap, d, seed):
    """A compact pool with `cap` slots per (b, g), its tables, and contiguous K/V of a long
    sequence per b to admit from."""
    g = torch.Generator().manual_seed(seed)
    mb = (cap + 15) // 16
    nb = B * mb + 3
    perm = torch.randperm(nb, generator=g)[: B * mb].view(B, mb).to(torch.int32)
    kc = np.zeros((nb, hkv, 16, d), dtype=np.uint16)
    vc = np.zeros((nb, hkv, 16, d), dtype=np.uint16)
    return kc, vc, perm.numpy()


def _slot_rows(kc, bt, b, g, s):
    return kc[bt[b, s // 16], g, s % 16]


@pytest.mark.parametrize("n_sink,k_top,n_recent", [(4, 24, 32), (1, 5, 7), (0, 16, 16), (4, 0, 20)])
def test_static_scores_keep_what_a_fresh_selection_keeps(n_sink, k_top, n_recent):
    B, hkv, d = 2, 3, 64
    cap = n_sink + k_top + n_recent
    L_final = 400
    rng = np.random.default_rng(cap)
    scores = rng.random((B, hkv, L_final)).astype(np.float32)  # distinct almost surely
    g = torch.Generator().manual_seed(cap + 1)
    K = rand_bf16((B, L_final, hkv, d), g)
    V = rand_bf16((B, L_final, hkv, d), g)
    kc, vc, bt = _pool(B, hkv, cap, d, seed=cap)
    pos = np.full((B, hkv, cap), -1, dtype=np.int32)
    sc = np.zeros((B, hkv, cap), dtype=np.float32)
    kl = np.zeros(B, dtype=np.int32)
    for L in range(1, L_final + 1):
        lens = np.full(B, L, dtype=np.int32)
        kc, vc, pos, sc, kl = oracle.rolling_admit(kc, vc, bt, pos, sc, kl, lens, bits(K[:, L - 1]),
                                                   bits(V[:, L - 1]), n_sink, n_recent)
        # the new token's score is fixed in advance (stands in for its accumulated score)
        for b in range(B):
            for h in range(hkv):
                s = int(np.nonzero(pos[b, h] == L - 1)[0][0])
                sc[b, h, s] = scores[b, h, L - 1]
    assert np.all(kl == cap)
    kept, kept_lens = oracle.select_topk(scores, np.full(B, L_final, dtype=np.int32), n_sink, n_recent, k_top)
    for b in range(B):
        for h in range(hkv):
            assert sorted(pos[b, h].tolist()) == kept[b, h, : kept_lens[b]].tolist()
            for s in range(cap):  # every slot holds the rows of the position it records
                p = pos[b, h, s]
                assert np.array_equal(_slot_rows(kc, bt, b, h, s), bits(K[b, p, h]))
                assert np.array_equal(_slot_rows(vc, bt, b, h, s), bits(V[b, p, h]))


def _full_state(positions, scores_list, cap, d=64):
    kc, vc, bt = _pool(1, 1, cap, d, seed=3)
    pos = np.array(positions, dtype=np.int32).reshape(1, 1, cap)
    sc = np.array(scores_list, dtype=np.float32).reshape(1, 1, cap)
    return kc, vc, bt, pos, sc, np.array([cap], dtype=np.int32)


def _admit(state, L, n_sink, n_recent):
    kc, vc, bt, pos, sc, kl = state
    k_new = np.full((1, 1, kc.shape[3]), 0x3F80, dtype=np.uint16)  # 1.0 in bf16
    return oracle.rolling_admit(kc, vc, bt, pos, sc, kl, np.array([L], np.int32), k_new, k_new, n_sink, n_recent)


def test_equal_lowest_scores_drop_the_highest_position():
    # sink 0; top-k {1, 5, 9}; recent {10, 11}; new token 12 -> token 10 leaves with score 0.9
    positions = [0, 5, 1, 9, 10, 11]
    scores_ = [9.0, 0.25, 0.25, 0.25, 0.9, 0.0]
    _, _, pos, sc, _ = _admit(_full_state(positions, scores_, 6), 13, 1, 2)
    assert sorted(pos[0, 0].tolist()) == [0, 1, 5, 10, 11, 12]   # 9 dropped, 10 joins the top-k
    assert pos[0, 0, 3] == 12 and sc[0, 0, 3] == 0.0              # the new token took 9's slot


def test_leaving_token_equal_to_the_lowest_is_dropped():
    positions = [0, 5, 1, 9, 10, 11]
    scores_ = [9.0, 0.25, 0.5, 0.5, 0.25, 0.0]
    _, _, pos, _, _ = _admit(_full_state(positions, scores_, 6), 13, 1, 2)
    assert sorted(pos[0, 0].tolist()) == [0, 1, 5, 9, 11, 12]
    assert pos[0, 0, 4] == 12                                      # 10's slot


def test_no_top_k_keeps_sinks_and_the_recent_window():
    state = _full_state([0, 1, 7, 8, 9], [1.0, 1.0, 5.0, 5.0, 5.0], 5)
    _, _, pos, _, _ = _admit(state, 11, 2, 3)                      # leaving 7 has no set to join
    assert sorted(pos[0, 0].tolist()) == [0, 1, 8, 9, 10]


def test_invalid_states_are_refused():
    state = _full_state([0, 5, 1, 9, 10, 11], [9.0, np.nan, 0.25, 0.25, 0.9, 0.0], 6)
    with pytest.raises(RuntimeError):
        _admit(state, 13, 1, 2)
    state = _full_state([0, 5, 1, 9, 4, 11], [9.0, 0.1, 0.25, 0.25, 0.9, 0.0], 6)  # 10 missing
    with pytest.raises(RuntimeError):
        _admit(state, 13, 1, 2)
