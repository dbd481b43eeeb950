"""Pins of the oracle's INT8 KV cache (oracle.quantize_rows, kv_append_q8, paged_decode_q8) to
facts outside it.

  Codes are checked as the pools store them: each code c as the byte c + 128.
  * exact round trips: a row whose values are integer codes times a power-of-two scale (one
    code of magnitude 127) quantizes back to exactly those codes and that scale;
  * hand-worked half-way ties (scale 1): round half to even;
  * the rounding bound |x - c s| <= s (1/2 + 2^-17) (half a step plus the fp32 quotient's
    rounding) and |c| <= 127 on random rows, the absmax element at +-127, zero rows at scale 0;
  * non-finite elements refused;
  * append: a dict-of-slots model, untouched rows unchanged;
  * decode over INT8 pools equals the bf16 decode bit for bit where every code * scale is a
    bf16 value, and matches torch SDPA (fp64) on the dequantized contiguous K/V otherwise.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import bits, code_values, from_bits, paged_from_contiguous, rand_bf16, stored_codes


def _bf16_bits_of(values: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(t.to(torch.float32), torch.from_numpy(np.asarray(values, dtype=np.float32))), \
        "test values must be bf16-exact"
    return bits(t)


def test_codes_times_power_of_two_round_trip_exactly():
    rng = np.random.default_rng(1)
    for d, e in ((64, -9), (128, -3), (128, 0), (64, 4)):
        codes = rng.integers(-127, 128, size=(20, d))
        codes[np.arange(20), rng.integers(0, d, size=20)] = rng.choice([-127, 127], size=20)
        x = codes.astype(np.float32) * np.float32(2.0 ** e)
        c, s = oracle.quantize_rows(_bf16_bits_of(x))
        assert c.dtype == np.uint8 and np.array_equal(code_values(c), codes)
        assert np.all(s == np.float32(2.0 ** e))


def test_half_way_ties_round_to_even():
    # amax 127 -> scale exactly 1, so x / s = x and the ties are exact
    row = [127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 126.5, -1.5, 1.0, 0.0]
    want = [127, 2, 4, -2, 0, 0, 126, -2, 1, 0]
    x = np.zeros((1, 16), dtype=np.float32)
    x[0, :len(row)] = row
    c, s = oracle.quantize_rows(_bf16_bits_of(x))
    assert s[0] == np.float32(1.0)
    assert code_values(c)[0, :len(want)].tolist() == want


def test_rounding_bound_and_absmax_code():
    g = torch.Generator().manual_seed(2)
    x = rand_bf16((64, 128), g) * torch.logspace(-6, 6, 64).view(-1, 1).to(torch.bfloat16)
    c, s = oracle.quantize_rows(bits(x))
    c = code_values(c)
    xf = x.to(torch.float64).numpy()
    deq = c.astype(np.float64) * s.astype(np.float64)[:, None]
    assert np.all(np.abs(c) <= 127)
    # half a step, plus the fp32 quotient's rounding (half an ulp of a value below 128: 2^-18)
    assert np.all(np.abs(xf - deq) <= s.astype(np.float64)[:, None] * (0.5 + 2.0 ** -17))
    amax_at = np.argmax(np.abs(xf), axis=1)
    assert np.all(np.abs(c[np.arange(64), amax_at].astype(np.int32)) == 127)
    # the scale is the absmax over 127 to within fp32 rounding
    np.testing.assert_allclose(s.astype(np.float64), np.abs(xf).max(axis=1) / 127.0, rtol=2 ** -23)


def test_zero_rows_and_non_finite_refused():
    c, s = oracle.quantize_rows(np.zeros((3, 64), dtype=np.uint16))
    assert np.all(code_values(c) == 0) and np.all(c == 128) and np.all(s == 0.0)
    for bad in (np.inf, -np.inf, np.nan):
        x = np.ones((2, 64), dtype=np.float32)
        x[1, 7] = bad
        xb = bits(torch.from_numpy(x).to(torch.bfloat16))
        with pytest.raises(oracle.OracleError):
            oracle.quantize_rows(xb)


def test_append_q8_writes_quantized_rows_at_their_slots():
    nb, hkv, d, T = 6, 3, 64, 9
    g = torch.Generator().manual_seed(3)
    rng = np.random.default_rng(3)
    kc = stored_codes(rng.integers(-127, 128, size=(nb, hkv, 16, d)))
    vc = stored_codes(rng.integers(-127, 128, size=(nb, hkv, 16, d)))
    ks = rng.random((nb, hkv, 16)).astype(np.float32)
    vs = rng.random((nb, hkv, 16)).astype(np.float32)
    k = bits(rand_bf16((T, hkv, d), g))
    v = bits(rand_bf16((T, hkv, d), g))
    slots = rng.choice(nb * 16, size=T, replace=False).astype(np.int64)
    slots[4] = -1
    kc2, vc2, ks2, vs2 = oracle.kv_append_q8(kc, vc, ks, vs, k, v, slots)
    written = {}
    for i, sl in enumerate(slots):
        if sl >= 0:
            written[(sl // 16, sl % 16)] = i
    for blk in range(nb):
        for off in range(16):
            i = written.get((blk, off))
            for h in range(hkv):
                if i is None:
                    assert np.array_equal(kc2[blk, h, off], kc[blk, h, off]) and ks2[blk, h, off] == ks[blk, h, off]
                    assert np.array_equal(vc2[blk, h, off], vc[blk, h, off]) and vs2[blk, h, off] == vs[blk, h, off]
                else:
                    ck, sk = oracle.quantize_rows(k[i, h][None])
                    cv, sv = oracle.quantize_rows(v[i, h][None])
                    assert np.array_equal(kc2[blk, h, off], ck[0]) and ks2[blk, h, off] == sk[0]
                    assert np.array_equal(vc2[blk, h, off], cv[0]) and vs2[blk, h, off] == sv[0]


def _pow2_q8_pools(nb, hkv, d, seed):
    """INT8 pools whose every code * scale is a bf16 value (scales are powers of two), and the
    bf16 pools holding those same values."""
    rng = np.random.default_rng(seed)
    pools = []
    for _ in range(2):
        codes = rng.integers(-127, 128, size=(nb, hkv, 16, d))
        scales = (2.0 ** rng.integers(-9, 2, size=(nb, hkv, 16))).astype(np.float32)
        vals = codes.astype(np.float32) * scales[..., None]
        pools.append((stored_codes(codes), scales, _bf16_bits_of(vals)))
    return pools


@pytest.mark.parametrize("hq,hkv,d,window", [(8, 2, 64, 0), (12, 2, 128, 0), (8, 8, 64, 37), (32, 8, 128, 0)])
def test_q8_decode_equals_bf16_decode_on_representable_values(hq, hkv, d, window):
    lens = [70, 1, 0, 33, 160]
    nb = 60
    (kc, ks, kb), (vc, vs, vb) = _pow2_q8_pools(nb, hkv, d, seed=hq + d)
    g = torch.Generator().manual_seed(hq * d)
    q = bits(rand_bf16((len(lens), hq, d), g))
    bt = torch.randperm(nb, generator=g)[: len(lens) * 10].view(len(lens), 10).to(torch.int32).numpy()
    L = np.array(lens, dtype=np.int32)
    got = oracle.paged_decode_q8(q, kc, ks, vc, vs, bt, L, d ** -0.5, window)
    ref = oracle.paged_decode(q, kb, vb, bt, L, d ** -0.5, window)
    assert np.array_equal(got, ref)


def test_q8_decode_matches_sdpa_on_dequantized_values():
    g = torch.Generator().manual_seed(4)
    lens = [90, 17, 64]
    B, hq, hkv, d = 3, 8, 2, 128
    k = rand_bf16((B, 90, hkv, d), g) * 3
    v = rand_bf16((B, 90, hkv, d), g)
    q = rand_bf16((B, hq, d), g)
    kc, vc, bt = paged_from_contiguous(k, v, lens, 20, g)
    kq, ks = oracle.quantize_rows(bits(kc))
    vq, vs = oracle.quantize_rows(bits(vc))
    ks[0, 0, 3] = 0.0  # a zero-scale row reads as zeros
    scale = d ** -0.5
    for window in (0, 20):
        got = oracle.paged_decode_q8(bits(q), kq, ks, vq, vs, bt.numpy(), np.array(lens, np.int32), scale, window)
        kd = torch.from_numpy(code_values(kq).astype(np.float64) * ks.astype(np.float64)[..., None])
        vd = torch.from_numpy(code_values(vq).astype(np.float64) * vs.astype(np.float64)[..., None])
        for b, L in enumerate(lens):
            s0 = max(0, L - window) if window else 0
            idx = torch.arange(s0, L)
            phys = bt[b, idx // 16].long()
            kk = kd[phys, :, idx % 16].permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)  # [Hq, n, d]
            vv = vd[phys, :, idx % 16].permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
            ref = torch.nn.functional.scaled_dot_product_attention(
                q[b].to(torch.float64)[:, None], kk, vv, scale=scale)[:, 0]
            np.testing.assert_allclose(got[b], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_quantized_decode_stays_near_the_bf16_decode():
    """Sanity of the reading (not a pin): with K/V rows of N(0,1), per-row INT8 moves the
    output by about the quantization step."""
    g = torch.Generator().manual_seed(5)
    lens = [300, 120]
    k = rand_bf16((2, 300, 2, 128), g)
    v = rand_bf16((2, 300, 2, 128), g)
    q = rand_bf16((2, 8, 128), g)
    kc, vc, bt = paged_from_contiguous(k, v, lens, 30, g)
    kq, ks = oracle.quantize_rows(bits(kc))
    vq, vs = oracle.quantize_rows(bits(vc))
    L = np.array(lens, np.int32)
    a = oracle.paged_decode_q8(bits(q), kq, ks, vq, vs, bt.numpy(), L, 128 ** -0.5)
    b = oracle.paged_decode(bits(q), bits(kc), bits(vc), bt.numpy(), L, 128 ** -0.5)
    assert np.abs(a - b).max() < 0.02
    assert from_bits(bits(q)).shape == q.shape
