"""Pins of the oracle's sparsification score (oracle.decode_scores) to facts outside it.

The score of (sequence b, kv head g, position t) after one decode step is the sum, over the
G query heads sharing kv head g, of each head's softmax probability of key t; the oracle also
returns every row's log-sum-exp.  Pinned by:
  * library routine: torch softmax / logsumexp in fp64 over the contiguous K (GQA by
    repeat_interleave), with and without a window;
  * invariants: each head's probabilities sum to 1, so a segment's scores sum to G; permuting
    physical blocks changes nothing; no score outside the attended window;
  * closed forms: q = 0 gives G / n on every attended key and lse = log n; one attended key
    gets G and lse = its logit; two keys get the logistic weights;
  * consistency with the attention output: sum_t p_t V_t reproduces the oracle's decode.
"""
import math

import numpy as np
import torch
from scipy.special import expit

import oracle
from helpers import bits, bf16_to_f64, paged_from_contiguous, rand_bf16


def _case(lens, hq, hkv, d, seed, nb_extra=3, q=None, k=None, v=None):
    g = torch.Generator().manual_seed(seed)
    B = len(lens)
    lmax = max(max(lens), 1)
    k = rand_bf16((B, lmax, hkv, d), g) if k is None else k
    v = rand_bf16((B, lmax, hkv, d), g) if v is None else v
    q = rand_bf16((B, hq, d), g) if q is None else q
    nb = sum((L + 15) // 16 for L in lens) + nb_extra
    kc, vc, bt = paged_from_contiguous(k, v, lens, nb, g)
    return dict(q=q, k=k, v=v, kc=kc, vc=vc, bt=bt, lens=torch.tensor(lens, dtype=torch.int32))


def _scores(c, scale, window=0, stride=None):
    return oracle.decode_scores(bits(c["q"]), bits(c["kc"]), c["bt"].numpy(), c["lens"].numpy(),
                                scale, window, stride=stride)


def _torch_ref(c, scale, window=0, stride=None):
    """softmax / logsumexp (fp64) over the contiguous keys, probabilities summed per group."""
    q, k, lens = c["q"], c["k"], c["lens"]
    B, hq, d = q.shape
    hkv = k.shape[2]
    G = hq // hkv
    stride = stride or max(int(lens.max()), 1)
    score = np.zeros((B, hkv, stride))
    lse = np.full((B, hq), -np.inf)
    for b in range(B):
        L = int(lens[b])
        s = max(0, L - window) if window > 0 else 0
        if L == 0:
            continue
        kk = k[b, s:L].to(torch.float64).permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq, n, d]
        logits = torch.einsum("hd,hnd->hn", q[b].to(torch.float64), kk) * scale
        p = torch.softmax(logits, dim=-1)
        lse[b] = torch.logsumexp(logits, dim=-1).numpy()
        score[b, :, s:L] = p.view(hkv, G, -1).sum(dim=1).numpy()
    return score, lse


def test_matches_torch_softmax_all_groups_and_windows():
    for hq, hkv, d in ((8, 8, 64), (8, 2, 64), (12, 2, 128), (16, 2, 64)):
        c = _case([37, 1, 0, 130, 16], hq, hkv, d, seed=hq * 100 + hkv)
        for window in (0, 1, 20, 200):
            got, lse = _scores(c, d ** -0.5, window)
            ref, ref_lse = _torch_ref(c, d ** -0.5, window)
            np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_scores_of_a_segment_sum_to_group_size():
    c = _case([300, 17, 64], 12, 2, 128, seed=3)
    got, _ = _scores(c, 0.09)
    np.testing.assert_allclose(got.sum(axis=2), np.full((3, 2), 6.0), rtol=1e-12)


def test_empty_context_zero_scores_and_minus_infinity_lse():
    c = _case([0, 5], 4, 2, 64, seed=4)
    got, lse = _scores(c, 0.125, stride=8)
    assert np.all(got[0] == 0.0) and np.all(np.isneginf(lse[0]))
    np.testing.assert_allclose(got[1].sum(axis=1), [2.0, 2.0], rtol=1e-12)


def test_q_zero_gives_uniform_scores_and_log_n():
    lens = [50, 7]
    c = _case(lens, 8, 2, 64, seed=5, q=torch.zeros(2, 8, 64, dtype=torch.bfloat16))
    got, lse = _scores(c, 0.3)
    for b, L in enumerate(lens):
        np.testing.assert_allclose(got[b, :, :L], 4.0 / L, rtol=1e-13)
        assert np.all(got[b, :, L:] == 0.0)
        np.testing.assert_allclose(lse[b], math.log(L), rtol=1e-13)


def test_single_key_gets_group_size_and_its_logit():
    c = _case([200], 8, 4, 64, seed=6)
    scale = 0.11
    got, lse = _scores(c, scale, window=1)
    assert np.all(got[0, :, :199] == 0.0)
    np.testing.assert_allclose(got[0, :, 199], 2.0, rtol=1e-14)
    q = bf16_to_f64(c["q"][0])                              # [Hq, d]
    k_last = bf16_to_f64(c["k"][0, 199])                    # [Hkv, d]
    logit = np.array([scale * float(q[h] @ k_last[h // 2]) for h in range(8)])
    np.testing.assert_allclose(lse[0], logit, rtol=1e-13, atol=1e-13)


def test_two_keys_logistic_weights():
    c = _case([2], 2, 1, 64, seed=7)
    scale = 0.2
    got, _ = _scores(c, scale)
    q = bf16_to_f64(c["q"][0])
    k = bf16_to_f64(c["k"][0, :, 0])                        # [2, d]
    exp0 = sum(expit(scale * (float(q[h] @ k[0]) - float(q[h] @ k[1]))) for h in range(2))
    np.testing.assert_allclose(got[0, 0, 0], exp0, rtol=1e-13)
    np.testing.assert_allclose(got[0, 0, 1], 2.0 - exp0, rtol=1e-13)


def test_block_permutation_changes_nothing():
    g = torch.Generator().manual_seed(8)
    lens = [90, 33]
    k = rand_bf16((2, 90, 2, 64), g)
    v = rand_bf16((2, 90, 2, 64), g)
    q = rand_bf16((2, 4, 64), g)
    a = oracle.decode_scores(bits(q), *(lambda kc, vc, bt: (bits(kc), bt.numpy()))(
        *paged_from_contiguous(k, v, lens, 20, torch.Generator().manual_seed(1))), np.array(lens, np.int32), 0.1)
    b = oracle.decode_scores(bits(q), *(lambda kc, vc, bt: (bits(kc), bt.numpy()))(
        *paged_from_contiguous(k, v, lens, 20, torch.Generator().manual_seed(2))), np.array(lens, np.int32), 0.1)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_probabilities_reproduce_the_attention_output():
    """sum_t p_{h,t} V_t (p from the group score with G = 1) equals the oracle's decode row."""
    c = _case([70, 3], 4, 4, 64, seed=9)
    scale = 0.125
    got, _ = _scores(c, scale)                              # G = 1: score = the head's p
    out = oracle.paged_decode(bits(c["q"]), bits(c["kc"]), bits(c["vc"]), c["bt"].numpy(),
                              c["lens"].numpy(), scale)
    for b, L in enumerate((70, 3)):
        v = bf16_to_f64(c["v"][b, :L])                      # [L, Hkv, d]
        recon = np.einsum("hl,lhd->hd", got[b, :, :L], v)
        np.testing.assert_allclose(recon, out[b], rtol=1e-11, atol=1e-12)


def test_segment_subset_matches_full_run():
    c = _case([40, 25, 9], 8, 2, 64, seed=10)
    full, full_lse = _scores(c, 0.1)
    segs = [5, 0, 3]
    sub, sub_lse = oracle.decode_scores(bits(c["q"]), bits(c["kc"]), c["bt"].numpy(), c["lens"].numpy(),
                                        0.1, segs=segs)
    for i, s in enumerate(segs):
        assert np.array_equal(sub[i], full[s // 2, s % 2])
        assert np.array_equal(sub_lse[i], full_lse[s // 2, (s % 2) * 4:(s % 2) * 4 + 4])
