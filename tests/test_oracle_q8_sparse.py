"""Pins of the oracle's INT8 sparse-layer functions (oracle.decode_scores_q8, compact_q8,
rolling_admit_q8) to facts outside them.

  * the score over INT8 K equals the bf16 score bit for bit where every code * scale is a
    bf16 value, and matches torch softmax (fp64) on the dequantized K otherwise; a zero-scale
    row has logit 0;
  * compaction: a dict-of-slots model (codes and row scales move together, untouched rows
    unchanged), and dequantize-then-compact == compact-then-dequantize;
  * rolling admission: the slot choice, positions, scores and counts of the bf16 admission on
    the same state, the admitted rows equal to quantize_rows of the new token, every other
    row unchanged; a non-finite new row refused;
  * sparse decode over INT8 pools: equal bit for bit to the bf16 sparse decode where every
    code * scale is a bf16 value, and to the INT8 paged decode when every token is kept.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import bits, code_values, paged_from_contiguous, rand_bf16, stored_codes


def _bf16_bits_of(values: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(t.to(torch.float32), torch.from_numpy(np.asarray(values, dtype=np.float32)))
    return bits(t)


def _pow2_pool(nb, hkv, d, rng):
    """INT8 codes (stored as code + 128) and power-of-two row scales, and the bf16 pool of the
    same values."""
    codes = rng.integers(-127, 128, size=(nb, hkv, 16, d))
    scales = (2.0 ** rng.integers(-9, 2, size=(nb, hkv, 16))).astype(np.float32)
    return stored_codes(codes), scales, _bf16_bits_of(codes.astype(np.float32) * scales[..., None])


def _dequant(stored, scales):
    return code_values(stored).astype(np.float64) * scales.astype(np.float64)[..., None]


@pytest.mark.parametrize("hq,hkv,d,window", [(8, 2, 64, 0), (12, 2, 128, 0), (8, 8, 64, 21), (32, 8, 128, 0)])
def test_scores_q8_equal_bf16_scores_on_representable_values(hq, hkv, d, window):
    rng = np.random.default_rng(hq + d + window)
    lens = np.array([70, 1, 0, 33, 150], dtype=np.int32)
    nb = 60
    kc, ks, kb = _pow2_pool(nb, hkv, d, rng)
    g = torch.Generator().manual_seed(hq * d)
    q = bits(rand_bf16((len(lens), hq, d), g))
    bt = torch.randperm(nb, generator=g)[: len(lens) * 10].view(len(lens), 10).to(torch.int32).numpy()
    s8, l8 = oracle.decode_scores_q8(q, kc, ks, bt, lens, d ** -0.5, window, stride=170)
    sb, lb = oracle.decode_scores(q, kb, bt, lens, d ** -0.5, window, stride=170)
    assert np.array_equal(s8, sb) and np.array_equal(l8, lb)


def test_scores_q8_match_torch_softmax_on_dequantized_k():
    g = torch.Generator().manual_seed(6)
    lens = [90, 17, 64]
    B, hq, hkv, d = 3, 8, 2, 128
    G = hq // hkv
    k = rand_bf16((B, 90, hkv, d), g) * 3
    q = rand_bf16((B, hq, d), g)
    kcache, _, bt = paged_from_contiguous(k, k, lens, 20, g)
    kq, ks = oracle.quantize_rows(bits(kcache))
    blk0 = int(bt[0, 0])
    ks[blk0, 1, 3] = 0.0  # token 3 of sequence 0, kv head 1: logit exactly 0
    scale = d ** -0.5
    for window in (0, 25):
        score, lse = oracle.decode_scores_q8(bits(q), kq, ks, bt.numpy(), np.array(lens, np.int32), scale, window,
                                             stride=96)
        kd = torch.from_numpy(_dequant(kq, ks))
        for b, L in enumerate(lens):
            s0 = max(0, L - window) if window else 0
            idx = torch.arange(s0, L)
            phys = bt[b, idx // 16].long()
            kk = kd[phys, :, idx % 16]  # [n, Hkv, d]
            for h in range(hq):
                gg = h // G
                logits = (kk[:, gg] @ q[b, h].to(torch.float64)) * scale
                if b == 0 and gg == 1 and window == 0:
                    assert logits[3].item() == 0.0
                np.testing.assert_allclose(lse[b, h], torch.logsumexp(logits, 0).item(), rtol=1e-13)
            for gg in range(hkv):
                want = np.zeros(96)
                for h in range(gg * G, gg * G + G):
                    logits = (kk[:, gg] @ q[b, h].to(torch.float64)) * scale
                    want[s0:L] += torch.softmax(logits, 0).numpy()
                np.testing.assert_allclose(score[b, gg], want, rtol=1e-12, atol=1e-15)


def _compact_case(rng, d, nb_src=40, nb_dst=24):
    B, hkv = 3, 2
    lens = np.array([100, 37, 0], dtype=np.int32)
    sk, sks, _ = _pow2_pool(nb_src, hkv, d, rng)
    sv, svs, _ = _pow2_pool(nb_src, hkv, d, rng)
    sbt = rng.permutation(nb_src)[: B * 8].reshape(B, 8).astype(np.int32)
    max_kept = 40
    kept = np.full((B, hkv, max_kept), -1, dtype=np.int32)
    kept_lens = np.array([40, 37, 0], dtype=np.int32)
    for b in range(B):
        for g in range(hkv):
            n = kept_lens[b]
            kept[b, g, :n] = np.sort(rng.choice(lens[b], size=n, replace=False)) if n else []
    dbt = rng.permutation(nb_dst)[: B * 3].reshape(B, 3).astype(np.int32)
    dk = stored_codes(rng.integers(-127, 128, size=(nb_dst, hkv, 16, d)))
    dv = stored_codes(rng.integers(-127, 128, size=(nb_dst, hkv, 16, d)))
    dks = rng.random((nb_dst, hkv, 16)).astype(np.float32)
    dvs = rng.random((nb_dst, hkv, 16)).astype(np.float32)
    return dict(dk=dk, dv=dv, dks=dks, dvs=dvs, dbt=dbt, sk=sk, sv=sv, sks=sks, svs=svs, sbt=sbt,
                lens=lens, kept=kept, kept_lens=kept_lens)


@pytest.mark.parametrize("d", [64, 128])
def test_compact_q8_dict_of_slots_model(d):
    c = _compact_case(np.random.default_rng(d), d)
    dk, dv, dks, dvs = oracle.compact_q8(c["dk"], c["dv"], c["dks"], c["dvs"], c["dbt"], c["sk"], c["sv"], c["sks"],
                                         c["svs"], c["sbt"], c["lens"], c["kept"], c["kept_lens"])
    written = {}
    B, hkv, _ = c["kept"].shape
    for b in range(B):
        for g in range(hkv):
            for j in range(c["kept_lens"][b]):
                t = c["kept"][b, g, j]
                written[(int(c["dbt"][b, j // 16]), g, j % 16)] = (int(c["sbt"][b, t // 16]), t % 16)
    for blk in range(dk.shape[0]):
        for g in range(hkv):
            for off in range(16):
                src = written.get((blk, g, off))
                for got, gs, old, olds, s, ss in ((dk, dks, c["dk"], c["dks"], c["sk"], c["sks"]),
                                                  (dv, dvs, c["dv"], c["dvs"], c["sv"], c["svs"])):
                    if src is None:
                        assert np.array_equal(got[blk, g, off], old[blk, g, off]) and gs[blk, g, off] == olds[blk, g, off]
                    else:
                        assert np.array_equal(got[blk, g, off], s[src[0], g, src[1]])
                        assert gs[blk, g, off] == ss[src[0], g, src[1]]


def test_compact_q8_commutes_with_dequantization():
    rng = np.random.default_rng(7)
    c = _compact_case(rng, 64)
    dk, dv, dks, dvs = oracle.compact_q8(c["dk"], c["dv"], c["dks"], c["dvs"], c["dbt"], c["sk"], c["sv"], c["sks"],
                                         c["svs"], c["sbt"], c["lens"], c["kept"], c["kept_lens"])
    # the bf16 compaction of the same values (destination pools: representable values too)
    dst_kb = _bf16_bits_of(np.zeros(c["dk"].shape, np.float32))
    dst_vb = _bf16_bits_of(np.zeros(c["dv"].shape, np.float32))
    sk_b = _bf16_bits_of(_dequant(c["sk"], c["sks"]).astype(np.float32))
    sv_b = _bf16_bits_of(_dequant(c["sv"], c["svs"]).astype(np.float32))
    kb, vb = oracle.compact(dst_kb, dst_vb, c["dbt"], sk_b, sv_b, c["sbt"], c["lens"], c["kept"], c["kept_lens"])
    kf = torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    vf = torch.from_numpy(vb.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for b in range(3):
        for j in range(c["kept_lens"][b]):
            blk, off = c["dbt"][b, j // 16], j % 16
            assert np.array_equal(_dequant(dk, dks)[blk, :, off], kf[blk, :, off])
            assert np.array_equal(_dequant(dv, dvs)[blk, :, off], vf[blk, :, off])


def test_compact_q8_refuses_a_kept_index_past_the_context():
    c = _compact_case(np.random.default_rng(8), 64)
    c["kept"][1, 0, 3] = 37  # L_1 = 37
    with pytest.raises(oracle.OracleError):
        oracle.compact_q8(c["dk"], c["dv"], c["dks"], c["dvs"], c["dbt"], c["sk"], c["sv"], c["sks"], c["svs"],
                          c["sbt"], c["lens"], c["kept"], c["kept_lens"])


def test_rolling_admit_q8_follows_the_bf16_admission():
    rng = np.random.default_rng(9)
    g = torch.Generator().manual_seed(9)
    B, hkv, d, cap, n_sink, n_recent = 3, 2, 64, 24, 2, 4
    nb = 10
    bt = rng.permutation(nb)[: B * 2].reshape(B, 2).astype(np.int32)
    kc = stored_codes(rng.integers(-127, 128, size=(nb, hkv, 16, d)))
    vc = stored_codes(rng.integers(-127, 128, size=(nb, hkv, 16, d)))
    ks = rng.random((nb, hkv, 16)).astype(np.float32)
    vs = rng.random((nb, hkv, 16)).astype(np.float32)
    kb = bits(rand_bf16((nb, hkv, 16, d), g))
    vb = bits(rand_bf16((nb, hkv, 16, d), g))
    pos = np.zeros((B, hkv, cap), np.int32)
    sc = np.zeros((B, hkv, cap), np.float32)
    kl = np.zeros(B, np.int32)
    lens = np.zeros(B, np.int32)
    for step in range(40):  # fills the budget, then rolls; scores keep changing
        lens += 1
        kn = bits(rand_bf16((B, hkv, d), g))
        vn = bits(rand_bf16((B, hkv, d), g))
        sc = sc + rng.integers(0, 4, size=sc.shape).astype(np.float32)  # ties are frequent
        out8 = oracle.rolling_admit_q8(kc, vc, ks, vs, bt, pos, sc, kl, lens, kn, vn, n_sink, n_recent)
        outb = oracle.rolling_admit(kb, vb, bt, pos, sc, kl, lens, kn, vn, n_sink, n_recent)
        kc2, vc2, ks2, vs2, pos8, sc8, kl8 = out8
        kb2, vb2, posb, scb, klb = outb
        assert np.array_equal(pos8, posb) and np.array_equal(sc8, scb) and np.array_equal(kl8, klb)
        changed_b = np.argwhere(np.any(kb2 != kb, axis=-1) | np.any(vb2 != vb, axis=-1))
        written = {(int(x), int(y), int(z)) for x, y, z in changed_b}
        for b in range(B):
            for gg in range(hkv):
                slot = int(np.argwhere(posb[b, gg] == lens[b] - 1)[0, 0])
                blk, off = int(bt[b, slot // 16]), slot % 16
                written.add((blk, gg, off))
                ck, sk = oracle.quantize_rows(kn[b, gg][None])
                cv, sv = oracle.quantize_rows(vn[b, gg][None])
                assert np.array_equal(kc2[blk, gg, off], ck[0]) and ks2[blk, gg, off] == sk[0]
                assert np.array_equal(vc2[blk, gg, off], cv[0]) and vs2[blk, gg, off] == sv[0]
        mask = np.ones((nb, hkv, 16), bool)
        for w in written:
            mask[w] = False
        assert np.array_equal(kc2[mask], kc[mask]) and np.array_equal(ks2[mask], ks[mask])
        assert np.array_equal(vc2[mask], vc[mask]) and np.array_equal(vs2[mask], vs[mask])
        kc, vc, ks, vs, pos, sc, kl = kc2, vc2, ks2, vs2, pos8, sc8, kl8
        kb, vb = kb2, vb2
    assert np.all(kl == cap)


def test_rolling_admit_q8_refuses_a_non_finite_row():
    B, hkv, d, cap = 1, 1, 64, 16
    kc = np.zeros((2, hkv, 16, d), np.uint8)
    ks = np.zeros((2, hkv, 16), np.float32)
    x = np.ones((B, hkv, d), np.float32)
    x[0, 0, 5] = np.inf
    kn = bits(torch.from_numpy(x).to(torch.bfloat16))
    vn = bits(torch.ones((B, hkv, d), dtype=torch.bfloat16))
    with pytest.raises(oracle.OracleError):
        oracle.rolling_admit_q8(kc, kc, ks, ks, np.array([[1]], np.int32), np.zeros((B, hkv, cap), np.int32),
                                np.zeros((B, hkv, cap), np.float32), np.zeros(B, np.int32), np.ones(B, np.int32),
                                kn, vn, 0, 1)


def _kept_lists(rng, lens, hkv, max_kept):
    B = len(lens)
    kept = np.full((B, hkv, max_kept), -1, dtype=np.int32)
    kl = np.array([min(L, max_kept) for L in lens], dtype=np.int32)
    for b in range(B):
        for g in range(hkv):
            kept[b, g, :kl[b]] = np.sort(rng.choice(lens[b], size=kl[b], replace=False)) if kl[b] else []
    return kept, kl


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 64), (32, 8, 128)])
def test_sparse_q8_equals_bf16_sparse_on_representable_values(hq, hkv, d):
    rng = np.random.default_rng(hq + d)
    lens = [70, 1, 0, 150]
    nb = 60
    kc, ks, kb = _pow2_pool(nb, hkv, d, rng)
    vc, vs, vb = _pow2_pool(nb, hkv, d, rng)
    g = torch.Generator().manual_seed(hq * d + 1)
    q = bits(rand_bf16((len(lens), hq, d), g))
    bt = torch.randperm(nb, generator=g)[: len(lens) * 10].view(len(lens), 10).to(torch.int32).numpy()
    kept, kl = _kept_lists(rng, lens, hkv, 40)
    L = np.array(lens, np.int32)
    got = oracle.sparse_decode_q8(q, kc, ks, vc, vs, bt, L, kept, kl, d ** -0.5)
    ref = oracle.sparse_decode(q, kb, vb, bt, L, kept, kl, d ** -0.5)
    assert np.array_equal(got, ref)


def test_sparse_q8_with_every_token_kept_equals_paged_q8():
    rng = np.random.default_rng(11)
    lens = [37, 64, 1]
    hq, hkv, d, nb = 8, 2, 64, 20
    kc = stored_codes(rng.integers(-127, 128, size=(nb, hkv, 16, d)))
    vc = stored_codes(rng.integers(-127, 128, size=(nb, hkv, 16, d)))
    ks = rng.random((nb, hkv, 16)).astype(np.float32)
    vs = rng.random((nb, hkv, 16)).astype(np.float32)
    g = torch.Generator().manual_seed(12)
    q = bits(rand_bf16((3, hq, d), g))
    bt = rng.permutation(nb)[:12].reshape(3, 4).astype(np.int32)
    max_kept = 64
    kept = np.full((3, hkv, max_kept), -1, dtype=np.int32)
    for b, L in enumerate(lens):
        kept[b, :, :L] = np.arange(L)
    L = np.array(lens, np.int32)
    got = oracle.sparse_decode_q8(q, kc, ks, vc, vs, bt, L, kept, L.copy(), d ** -0.5)
    ref = oracle.paged_decode_q8(q, kc, ks, vc, vs, bt, L, d ** -0.5)
    assert np.array_equal(got, ref)
