"""Pins of the oracle's decode attention (paged and sparse) to facts outside the oracle.

Each case builds its paged pool by scattering contiguous K/V (tests/helpers.py), so the
expected value is stated on the contiguous data:
  * closed forms: q = 0 gives the mean of V; one token gives its V row; equal V rows give
    that row; two tokens give the logistic weighting; window 1 gives the last V row;
  * invariants: window >= L equals no window; permuting physical blocks changes nothing;
  * library routine: torch SDPA in fp64 on the contiguous K/V (GQA by repeat_interleave);
  * sparse: kept = everything equals paged; gather over the full pool equals paged decode
    over a compacted pool; SDPA over the contiguous kept rows.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import expit

import oracle
from helpers import bits, bf16_to_f64, paged_from_contiguous, rand_bf16


def _case(lens, hq, hkv, d, seed, nb_extra=3, fill=None, q=None, k=None, v=None):
    g = torch.Generator().manual_seed(seed)
    B = len(lens)
    lmax = max(max(lens), 1)
    k = rand_bf16((B, lmax, hkv, d), g) if k is None else k
    v = rand_bf16((B, lmax, hkv, d), g) if v is None else v
    q = rand_bf16((B, hq, d), g) if q is None else q
    nb = sum((L + 15) // 16 for L in lens) + nb_extra
    kc, vc, bt = paged_from_contiguous(k, v, lens, nb, g, fill=fill)
    return dict(q=q, k=k, v=v, kc=kc, vc=vc, bt=bt, lens=torch.tensor(lens, dtype=torch.int32))


def _run(c, scale, window=0):
    return oracle.paged_decode(bits(c["q"]), bits(c["kc"]), bits(c["vc"]), c["bt"].numpy(),
                               c["lens"].numpy(), scale, window)


def _sdpa(c, scale, window=0):
    """Contiguous reference: torch SDPA (fp64) per sequence over its last tokens."""
    q, k, v, lens = c["q"], c["k"], c["v"], c["lens"]
    B, hq, d = q.shape
    hkv = k.shape[2]
    out = np.zeros((B, hq, d))
    for b in range(B):
        L = int(lens[b])
        s = max(0, L - window) if window > 0 else 0
        if L == 0:
            continue
        kk = k[b, s:L].to(torch.float64).permute(1, 0, 2)          # [Hkv, n, d]
        vv = v[b, s:L].to(torch.float64).permute(1, 0, 2)
        kk = kk.repeat_interleave(hq // hkv, dim=0)                # [Hq, n, d]
        vv = vv.repeat_interleave(hq // hkv, dim=0)
        qq = q[b].to(torch.float64).unsqueeze(1)                   # [Hq, 1, d]
        o = F.scaled_dot_product_attention(qq, kk, vv, scale=scale)
        out[b] = o[:, 0, :].numpy()
    return out


def test_q_zero_gives_mean_of_v():
    c = _case([37, 5], hq=4, hkv=2, d=64, seed=1)
    c["q"] = torch.zeros_like(c["q"])
    got = _run(c, 0.125)
    for b, L in enumerate([37, 5]):
        vmean = bf16_to_f64(c["v"][b, :L]).mean(axis=0)            # [Hkv, d]
        for h in range(4):
            np.testing.assert_allclose(got[b, h], vmean[h // 2], rtol=0, atol=1e-12)


def test_zero_scale_gives_mean_of_v():
    c = _case([50], hq=2, hkv=1, d=64, seed=2)
    got = _run(c, 0.0)
    vmean = bf16_to_f64(c["v"][0, :50]).mean(axis=0)
    np.testing.assert_allclose(got[0, 1], vmean[0], rtol=0, atol=1e-12)


def test_single_token_gives_its_v_exactly():
    c = _case([1, 1], hq=8, hkv=8, d=128, seed=3)
    got = _run(c, 1 / np.sqrt(128))
    ref = bf16_to_f64(c["v"][:, 0])                               # [B, Hkv, d]
    assert np.array_equal(got, ref)


def test_equal_v_rows_give_that_row():
    g = torch.Generator().manual_seed(4)
    row = rand_bf16((1, 1, 2, 64), g)
    v = row.expand(1, 300, 2, 64).clone()
    c = _case([300], hq=4, hkv=2, d=64, seed=4, v=v)
    got = _run(c, 0.3)
    for h in range(4):
        np.testing.assert_allclose(got[0, h], bf16_to_f64(row[0, 0, h // 2]), rtol=1e-13, atol=0)


def test_two_tokens_logistic_weights():
    c = _case([2], hq=3, hkv=1, d=64, seed=5)
    scale = 0.2
    got = _run(c, scale)
    q = bf16_to_f64(c["q"][0])
    k = bf16_to_f64(c["k"][0, :2, 0])
    v = bf16_to_f64(c["v"][0, :2, 0])
    for h in range(3):
        s1, s2 = scale * q[h] @ k[0], scale * q[h] @ k[1]
        ref = expit(s1 - s2) * v[0] + expit(s2 - s1) * v[1]
        np.testing.assert_allclose(got[0, h], ref, rtol=1e-12, atol=1e-14)


def test_window_one_gives_last_v():
    c = _case([100, 17, 16], hq=4, hkv=4, d=64, seed=6)
    got = _run(c, 0.125, window=1)
    for b, L in enumerate([100, 17, 16]):
        assert np.array_equal(got[b], bf16_to_f64(c["v"][b, L - 1]))


def test_window_at_least_length_equals_full():
    c = _case([100, 33], hq=4, hkv=2, d=64, seed=7)
    full = _run(c, 0.125)
    assert np.array_equal(_run(c, 0.125, window=100), full)
    assert np.array_equal(_run(c, 0.125, window=5000), full)
    assert not np.array_equal(_run(c, 0.125, window=99), full)


def test_block_permutation_invariance():
    c = _case([70, 130, 16], hq=4, hkv=2, d=64, seed=8, nb_extra=10)
    ref = _run(c, 0.125)
    g = torch.Generator().manual_seed(80)
    nb = c["kc"].shape[0]
    perm = torch.randperm(nb, generator=g)          # new physical id of old block i = perm[i]
    kc2 = torch.empty_like(c["kc"])
    vc2 = torch.empty_like(c["vc"])
    kc2[perm] = c["kc"]
    vc2[perm] = c["vc"]
    bt2 = c["bt"].clone()
    valid = bt2 >= 0
    bt2[valid] = perm[bt2[valid].long()].to(torch.int32)
    c2 = dict(c, kc=kc2, vc=vc2, bt=bt2)
    assert np.array_equal(_run(c2, 0.125), ref)


def test_empty_context_gives_zero_row():
    c = _case([0, 20], hq=2, hkv=1, d=64, seed=9)
    got = _run(c, 0.125)
    assert np.all(got[0] == 0.0)
    assert np.any(got[1] != 0.0)


@pytest.mark.parametrize("lens,hq,hkv,d,window", [
    ([1, 15, 16, 17], 4, 4, 64, 0),
    ([100, 256], 8, 8, 64, 0),
    ([300, 45], 8, 2, 128, 0),
    ([299, 161], 6, 1, 128, 0),
    ([200, 31], 8, 2, 128, 50),
    ([64, 65], 4, 2, 64, 16),
])
def test_matches_sdpa_on_contiguous(lens, hq, hkv, d, window):
    c = _case(lens, hq, hkv, d, seed=sum(lens) + hq)
    scale = 1 / np.sqrt(d)
    np.testing.assert_allclose(_run(c, scale, window), _sdpa(c, scale, window), rtol=1e-10,
                               atol=1e-12)


def test_large_sink_logits_match_sdpa():
    g = torch.Generator().manual_seed(10)
    k = torch.randn((1, 200, 2, 128), generator=g)
    k[:, :2] *= 20.0
    c = _case([200], hq=8, hkv=2, d=128, seed=10, k=k.to(torch.bfloat16))
    scale = 1 / np.sqrt(128)
    np.testing.assert_allclose(_run(c, scale), _sdpa(c, scale), rtol=1e-10, atol=1e-12)


def test_unused_slots_never_read():
    c = _case([20, 35], hq=4, hkv=2, d=64, seed=11, fill=float("nan"))
    got = _run(c, 0.125)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, _sdpa(c, 0.125), rtol=1e-10, atol=1e-12)


def test_bad_block_id_is_refused():
    c = _case([40], hq=2, hkv=1, d=64, seed=12)
    c["bt"][0, 1] = c["kc"].shape[0]
    with pytest.raises(oracle.OracleError):
        _run(c, 0.125)


# ---------------------------------------------------------------------------------- sparse

def _sparse(c, kept, kept_lens, scale):
    return oracle.sparse_decode(bits(c["q"]), bits(c["kc"]), bits(c["vc"]), c["bt"].numpy(),
                                c["lens"].numpy(), kept, kept_lens, scale)


def test_sparse_all_kept_equals_paged():
    lens = [77, 160]
    c = _case(lens, hq=4, hkv=2, d=64, seed=20)
    kept = np.full((2, 2, 200), -1, dtype=np.int32)
    for b, L in enumerate(lens):
        kept[b, :, :L] = np.arange(L)
    got = _sparse(c, kept, np.array(lens, dtype=np.int32), 0.125)
    assert np.array_equal(got, _run(c, 0.125))


def test_sparse_matches_sdpa_on_kept_rows():
    lens = [150, 90]
    c = _case(lens, hq=4, hkv=2, d=64, seed=21)
    rng = np.random.default_rng(21)
    n = 40
    kept = np.zeros((2, 2, n), dtype=np.int32)
    for b, L in enumerate(lens):
        for gh in range(2):
            kept[b, gh] = np.sort(rng.choice(L, size=n, replace=False))
    got = _sparse(c, kept, np.array([n, n], dtype=np.int32), 0.125)
    for b in range(2):
        for h in range(4):
            gh = h // 2
            kk = c["k"][b, kept[b, gh], gh].to(torch.float64)[None]
            vv = c["v"][b, kept[b, gh], gh].to(torch.float64)[None]
            qq = c["q"][b, h].to(torch.float64)[None, None]
            ref = F.scaled_dot_product_attention(qq, kk, vv, scale=0.125)[0, 0].numpy()
            np.testing.assert_allclose(got[b, h], ref, rtol=1e-10, atol=1e-12)


def test_sparse_gather_equals_compacted_paged():
    lens = [300, 180]
    c = _case(lens, hq=8, hkv=2, d=128, seed=22)
    rng = np.random.default_rng(22)
    n = 52
    kept = np.zeros((2, 2, n), dtype=np.int32)
    for b, L in enumerate(lens):
        for gh in range(2):
            kept[b, gh] = np.sort(rng.choice(L, size=n, replace=False))
    kl = np.array([n, n], dtype=np.int32)
    scale = 1 / np.sqrt(128)
    gathered = _sparse(c, kept, kl, scale)
    per_seq = (n + 15) // 16
    nb = 2 * per_seq + 1
    dbt = np.array(np.random.default_rng(5).permutation(nb)[:2 * per_seq].reshape(2, per_seq),
                   dtype=np.int32)
    dk = np.zeros((nb, 2, 16, 128), dtype=np.uint16)
    dv = np.zeros((nb, 2, 16, 128), dtype=np.uint16)
    dk, dv = oracle.compact(dk, dv, dbt, bits(c["kc"]), bits(c["vc"]), c["bt"].numpy(),
                            c["lens"].numpy(), kept, kl)
    compact_out = oracle.paged_decode(bits(c["q"]), dk, dv, dbt, kl, scale)
    assert np.array_equal(gathered, compact_out)


def test_sparse_refuses_unsorted_or_out_of_range():
    c = _case([50], hq=2, hkv=1, d=64, seed=23)
    kept = np.array([[[3, 2, 9]]], dtype=np.int32)
    with pytest.raises(oracle.OracleError):
        _sparse(c, kept, np.array([3], dtype=np.int32), 0.125)
    kept = np.array([[[3, 9, 50]]], dtype=np.int32)
    with pytest.raises(oracle.OracleError):
        _sparse(c, kept, np.array([3], dtype=np.int32), 0.125)


def test_row_subset_matches_full():
    c = _case([90, 40, 130], hq=8, hkv=2, d=64, seed=24)
    full = _run(c, 0.125)
    rows = [0, 7, 9, 23]
    sub = oracle.paged_decode(bits(c["q"]), bits(c["kc"]), bits(c["vc"]), c["bt"].numpy(),
                              c["lens"].numpy(), 0.125, 0, rows=rows)
    for i, r in enumerate(rows):
        assert np.array_equal(sub[i], full[r // 8, r % 8])
