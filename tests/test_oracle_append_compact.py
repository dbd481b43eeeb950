"""Pins of the oracle's append and compaction against brute-force dict-of-slots models."""
import numpy as np
import pytest
import torch

import oracle
from helpers import bits

BLOCK = 16


def _pool(nb, hkv, d, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 1 << 16, size=(nb, hkv, BLOCK, d), dtype=np.uint16)


def test_append_matches_slot_dict():
    nb, hkv, d, T = 9, 3, 64, 20
    kc, vc = _pool(nb, hkv, d, 1), _pool(nb, hkv, d, 2)
    rng = np.random.default_rng(3)
    k = rng.integers(0, 1 << 16, size=(T, hkv, d), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(T, hkv, d), dtype=np.uint16)
    slots = rng.choice(nb * BLOCK, size=T, replace=False).astype(np.int64)
    slots[[2, 7]] = -1
    nk, nv = oracle.kv_append(kc, vc, k, v, slots)
    written = {int(s): i for i, s in enumerate(slots) if s >= 0}
    for slot in range(nb * BLOCK):
        blk, off = divmod(slot, BLOCK)
        for g in range(hkv):
            if slot in written:
                assert np.array_equal(nk[blk, g, off], k[written[slot], g])
                assert np.array_equal(nv[blk, g, off], v[written[slot], g])
            else:
                assert np.array_equal(nk[blk, g, off], kc[blk, g, off])
                assert np.array_equal(nv[blk, g, off], vc[blk, g, off])


def test_append_refuses_out_of_pool_slot():
    kc = _pool(2, 1, 64, 4)
    k = np.zeros((1, 1, 64), dtype=np.uint16)
    with pytest.raises(oracle.OracleError):
        oracle.kv_append(kc, kc, k, k, np.array([2 * BLOCK], dtype=np.int64))


def test_compact_matches_slot_dict():
    B, hkv, d = 2, 2, 64
    lens = np.array([70, 45], dtype=np.int32)
    src_nb = 12
    sk, sv = _pool(src_nb, hkv, d, 5), _pool(src_nb, hkv, d, 6)
    rng = np.random.default_rng(7)
    perm = rng.permutation(src_nb).astype(np.int32)
    sbt = np.full((B, 5), -1, dtype=np.int32)
    sbt[0, :5] = perm[:5]
    sbt[1, :3] = perm[5:8]
    max_kept, n = 24, np.array([20, 17], dtype=np.int32)
    kept = np.full((B, hkv, max_kept), -1, dtype=np.int32)
    for b in range(B):
        for g in range(hkv):
            kept[b, g, :n[b]] = np.sort(rng.choice(int(lens[b]), size=int(n[b]), replace=False))
    dst_nb = 5
    dbt = np.array([[3, 0], [4, 1]], dtype=np.int32)
    dk, dv = _pool(dst_nb, hkv, d, 8), _pool(dst_nb, hkv, d, 9)
    nk, nv = oracle.compact(dk, dv, dbt, sk, sv, sbt, lens, kept, n)
    expect = {}
    for b in range(B):
        for g in range(hkv):
            for j in range(int(n[b])):
                t = int(kept[b, g, j])
                src = (int(sbt[b, t // BLOCK]), g, t % BLOCK)
                dst = (int(dbt[b, j // BLOCK]), g, j % BLOCK)
                expect[dst] = src
    for blk in range(dst_nb):
        for g in range(hkv):
            for off in range(BLOCK):
                if (blk, g, off) in expect:
                    sb, sg, so = expect[(blk, g, off)]
                    assert np.array_equal(nk[blk, g, off], sk[sb, sg, so])
                    assert np.array_equal(nv[blk, g, off], sv[sb, sg, so])
                else:
                    assert np.array_equal(nk[blk, g, off], dk[blk, g, off])
                    assert np.array_equal(nv[blk, g, off], dv[blk, g, off])


def test_bf16_bits_roundtrip():
    t = torch.randn(3, 5).to(torch.bfloat16)
    b = bits(t)
    assert b.dtype == np.uint16 and b.shape == (3, 5)
    back = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)
    assert torch.equal(back, t)
