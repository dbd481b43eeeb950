"""Pins of the oracle's prefill-window score (oracle.prefill_scores) to facts outside it.

The score of key i in kv head g is the sum, over the last alpha prompt positions j >= i and the
G query heads of the group, of the causal softmax probability A[j][i].  Pinned by:
  * library routine: torch softmax (fp64) over causally masked logits of contiguous K;
  * invariants: every window row's probabilities sum to 1, so a segment's scores sum to G times
    the number of window rows; permuting physical blocks changes nothing;
  * closed form: q = 0 gives A[j][i] = 1 / (j + 1);
  * alpha = 1 is one decode step's score (oracle.decode_scores, itself pinned) of the last query;
  * given lse: handing back the computed lse reproduces the scores; lse + c scales them by e^-c.
"""
import math

import numpy as np
import torch

import oracle
from helpers import bits, paged_from_contiguous, rand_bf16


def _case(lens, alpha, hq, hkv, d, seed, zero_q=False, nb_extra=3):
    g = torch.Generator().manual_seed(seed)
    B = len(lens)
    lmax = max(max(lens), 1)
    k = rand_bf16((B, lmax, hkv, d), g)
    v = rand_bf16((B, lmax, hkv, d), g)
    q = torch.zeros((B, alpha, hq, d), dtype=torch.bfloat16) if zero_q else rand_bf16((B, alpha, hq, d), g)
    nb = sum((L + 15) // 16 for L in lens) + nb_extra
    kc, vc, bt = paged_from_contiguous(k, v, lens, nb, g)
    return dict(q=q, k=k, kc=kc, bt=bt, lens=torch.tensor(lens, dtype=torch.int32), alpha=alpha)


def _scores(c, scale, lse=None, stride=None):
    return oracle.prefill_scores(bits(c["q"]), bits(c["kc"]), c["bt"].numpy(), c["lens"].numpy(), c["alpha"],
                                 scale, lse=lse, stride=stride)


def _torch_ref(c, scale, stride):
    q, k, lens, alpha = c["q"], c["k"], c["lens"], c["alpha"]
    B, _, hq, d = q.shape
    hkv = k.shape[2]
    G = hq // hkv
    score = np.zeros((B, hkv, stride))
    lse = np.full((B, hq, alpha), -np.inf)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        kk = k[b, :L].to(torch.float64).permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq, L, d]
        pos = torch.arange(L - alpha, L)                                              # window positions
        qq = q[b].to(torch.float64).permute(1, 0, 2)                                  # [Hq, alpha, d]
        logits = torch.einsum("had,hld->hal", qq, kk) * scale
        mask = torch.arange(L).view(1, -1) > pos.view(-1, 1)                          # key after the row
        logits = logits.masked_fill(mask.view(1, alpha, L), float("-inf"))
        used = pos >= 0
        p = torch.softmax(logits[:, used], dim=-1)                                     # [Hq, used, L]
        lse[b][:, used.numpy()] = torch.logsumexp(logits[:, used], dim=-1).numpy()
        score[b, :, :L] = p.sum(dim=1).view(hkv, G, L).sum(dim=1).numpy()
    return score, lse


def test_matches_torch_causal_softmax():
    for hq, hkv, d, alpha in ((8, 2, 64, 16), (12, 2, 128, 40), (8, 8, 64, 1), (32, 8, 64, 33)):
        c = _case([90, 17, 130, 5, 1], alpha, hq, hkv, d, seed=hq + alpha)
        got, lse = _scores(c, d ** -0.5, stride=136)
        ref, ref_lse = _torch_ref(c, d ** -0.5, 136)
        np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_scores_sum_to_group_times_window_rows():
    lens = [300, 20, 64]
    alpha = 32
    c = _case(lens, alpha, 12, 2, 128, seed=3)
    got, _ = _scores(c, 0.09)
    rows = np.array([min(L, alpha) for L in lens], dtype=np.float64)
    np.testing.assert_allclose(got.sum(axis=2), np.repeat((6.0 * rows)[:, None], 2, axis=1), rtol=1e-12)


def test_q_zero_closed_form():
    lens = [50, 7]
    alpha = 10
    c = _case(lens, alpha, 8, 2, 64, seed=5, zero_q=True)
    got, lse = _scores(c, 0.3)
    for b, L in enumerate(lens):
        want = np.zeros(got.shape[2])
        for j in range(max(0, L - alpha), L):
            want[: j + 1] += 4.0 / (j + 1)
        np.testing.assert_allclose(got[b, 0], want, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(got[b, 1], want, rtol=1e-13, atol=1e-15)
        used = [r for r in range(alpha) if L - alpha + r >= 0]
        np.testing.assert_allclose(lse[b][:, used], np.log(np.array([L - alpha + r + 1 for r in used], float))[None]
                                   .repeat(8, 0), rtol=1e-13)


def test_alpha_one_is_the_decode_score_of_the_last_query():
    lens = [77, 160, 3]
    c = _case(lens, 1, 16, 4, 128, seed=7)
    got, lse = _scores(c, 0.1, stride=160)
    dec, dec_lse = oracle.decode_scores(bits(c["q"][:, 0]), bits(c["kc"]), c["bt"].numpy(), c["lens"].numpy(), 0.1,
                                        stride=160)
    np.testing.assert_allclose(got, dec, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse[:, :, 0], dec_lse, rtol=1e-13)


def test_given_lse_reproduces_and_shifts():
    c = _case([120, 45], 24, 8, 2, 64, seed=9)
    got, lse = _scores(c, 0.125)
    again, lse2 = _scores(c, 0.125, lse=lse)
    np.testing.assert_allclose(again, got, rtol=1e-14, atol=1e-16)
    assert np.array_equal(lse2, lse)
    shifted, _ = _scores(c, 0.125, lse=lse + 0.75)
    np.testing.assert_allclose(shifted, got * math.exp(-0.75), rtol=1e-13, atol=1e-16)


def test_block_permutation_changes_nothing():
    g = torch.Generator().manual_seed(11)
    lens = [90, 33]
    k = rand_bf16((2, 90, 2, 64), g)
    v = rand_bf16((2, 90, 2, 64), g)
    q = rand_bf16((2, 12, 4, 64), g)
    outs = []
    for seed in (1, 2):
        kc, _, bt = paged_from_contiguous(k, v, lens, 20, torch.Generator().manual_seed(seed))
        outs.append(oracle.prefill_scores(bits(q), bits(kc), bt.numpy(), np.array(lens, np.int32), 12, 0.1))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
