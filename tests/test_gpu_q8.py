"""GPU parity of the INT8 KV cache: the quantized append (pkv_kv_append_q8) bit for bit against
oracle.kv_append_q8, and the decode over INT8 pools (pkv_paged_decode_attention_q8) against the
fp64 oracle.paged_decode_q8 (values code * scale), with the decode's max-abs / rel-L2 gate
applied to outputs divided by max(1, max |ref|): the gate's absolute part is meant for outputs
of unit scale, and bf16 output rounding alone (half an ulp) exceeds it once outputs pass 2."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_mapped_gb300 as pkv
from paged_kv_cache_mapped_gb300 import inputs as W
from helpers import assert_attn_close, bits, code_values, paged_from_contiguous, rand_bf16, stored_codes

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _q8_of(kc, vc):
    """INT8 pools (device) quantized by the oracle from bf16 pools."""
    kq, ks = oracle.quantize_rows(bits(kc))
    vq, vs = oracle.quantize_rows(bits(vc))
    t = lambda a: torch.from_numpy(a).to(DEV)
    return t(kq), t(ks), t(vq), t(vs)


def _case(lens, hq, hkv, d, seed, kmul=1.0, vmul=None):
    g = torch.Generator().manual_seed(seed)
    B = len(lens)
    lmax = max(max(lens), 1)
    k = rand_bf16((B, lmax, hkv, d), g) * kmul
    v = rand_bf16((B, lmax, hkv, d), g)
    if vmul is not None:
        v = (v.float() * vmul.view(1, -1, 1, 1)[:, :lmax]).to(torch.bfloat16)
    q = rand_bf16((B, hq, d), g)
    nb = sum((L + 15) // 16 for L in lens) + 5
    kc, vc, bt = paged_from_contiguous(k, v, lens, nb, g)
    kq, ks, vq, vs = _q8_of(kc, vc)
    return {"q": q.to(DEV), "kq": kq, "ks": ks, "vq": vq, "vs": vs, "bt": bt.to(DEV),
            "lens": torch.tensor(lens, dtype=torch.int32, device=DEV), "scale": d ** -0.5}


def _gpu(c, window=0, err=None, **kw):
    out = pkv.paged_decode_attention_q8(c["q"], c["kq"], c["vq"], c["ks"], c["vs"], c["bt"], c["lens"], c["scale"],
                                        window, error_word=err, **kw)
    torch.cuda.synchronize()
    return out


def _close(got, ref, what):
    top = max(1.0, float(np.abs(ref).max()) if ref.size else 1.0)
    assert_attn_close(got.float() / top, ref / top, what)


def _ref(c, window=0, rows=None):
    n = lambda t: t.cpu().numpy()
    return oracle.paged_decode_q8(bits(c["q"]), n(c["kq"]), n(c["ks"]), n(c["vq"]), n(c["vs"]), n(c["bt"]),
                                  n(c["lens"]), c["scale"], window, rows=rows)


@pytest.mark.parametrize("d", [64, 128])
def test_append_q8_bit_exact(d):
    nb, hkv, T = 40, 4, 300
    g = torch.Generator().manual_seed(d)
    rng = np.random.default_rng(d)
    k = rand_bf16((T, hkv, d), g) * torch.logspace(-3, 3, T).view(-1, 1, 1).to(torch.bfloat16)
    v = rand_bf16((T, hkv, d), g)
    # half-way ties: amax 127 gives scale 1, and k + 0.5 values sit exactly between codes
    tie = torch.arange(d, dtype=torch.float32) % 20 - 9.5
    tie[0] = 127.0
    k[5, 1] = tie.to(torch.bfloat16)
    k[6, 2] = 0.0                                  # a zero row
    slots = torch.from_numpy(rng.choice(nb * 16, size=T, replace=False).astype(np.int64))
    slots[7] = -1
    kq0 = torch.from_numpy(stored_codes(rng.integers(-127, 128, size=(nb, hkv, 16, d))))
    vq0 = torch.from_numpy(stored_codes(rng.integers(-127, 128, size=(nb, hkv, 16, d))))
    ks0 = torch.rand((nb, hkv, 16), generator=g)
    vs0 = torch.rand((nb, hkv, 16), generator=g)
    ref = oracle.kv_append_q8(kq0.numpy(), vq0.numpy(), ks0.numpy(), vs0.numpy(), bits(k), bits(v), slots.numpy())
    kq, vq, ks, vs = (t.to(DEV) for t in (kq0, vq0, ks0, vs0))
    err = pkv.new_error_word(DEV)
    pkv.kv_append_q8(kq, vq, ks, vs, k.to(DEV), v.to(DEV), slots.to(DEV), error_word=err)
    assert pkv.read_error(err) == 0
    for name, got, want in zip(("k_codes", "v_codes", "k_scales", "v_scales"), (kq, vq, ks, vs), ref):
        assert np.array_equal(got.cpu().numpy(), want), name


def test_append_q8_non_finite_reported_and_skipped():
    nb, hkv, d = 4, 2, 64
    k = torch.ones((3, hkv, d), dtype=torch.bfloat16)
    v = torch.ones((3, hkv, d), dtype=torch.bfloat16)
    v[1, 0, 9] = float("inf")
    slots = torch.tensor([0, 17, 33], dtype=torch.int64)
    kq = torch.zeros((nb, hkv, 16, d), dtype=torch.uint8, device=DEV)
    vq = torch.zeros_like(kq)
    ks = torch.full((nb, hkv, 16), 7.0, device=DEV)
    vs = torch.full((nb, hkv, 16), 7.0, device=DEV)
    err = pkv.new_error_word(DEV)
    pkv.kv_append_q8(kq, vq, ks, vs, k.to(DEV), v.to(DEV), slots.to(DEV), error_word=err)
    assert pkv.read_error(err) == pkv.header_constants()["PKV_DEV_BAD_VALUE"]
    assert ks[1, 0, 1].item() == 7.0 and torch.all(kq[1, 0, 1] == 0)     # token 1, kv head 0 skipped
    # written rows of ones: code 127 everywhere, stored as the byte 255
    assert ks[1, 1, 1].item() == pytest.approx(1 / 127) and np.all(code_values(kq[1, 1, 1]) == 127)  # head 1
    assert np.all(code_values(kq[0, :, 0]) == 127) and np.all(code_values(kq[2, :, 1]) == 127)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("group", [1, 4, 6, 8])
def test_ragged_lengths_all_groups(d, group):
    hkv = 2
    c = _case([700, 1, 0, 33, 1500, 16, 257], hkv * group, hkv, d, seed=d + group)
    _close(_gpu(c), _ref(c), f"d={d} G={group}")


@pytest.mark.parametrize("window", [1, 16, 50, 300])
def test_windows(window):
    c = _case([900, 70, 301], 16, 4, 128, seed=window)
    _close(_gpu(c, window), _ref(c, window), f"window={window}")


def test_v_scales_spanning_many_decades():
    """V rows whose scales grow and shrink by 10^6 along the sequence: the V-scale reference
    moves (and rescales the output) many times, and tiny rows still count."""
    lens = [1200, 640]
    ramp = torch.cat([torch.logspace(-3, 3, 600), torch.logspace(3, -3, 600)])
    c = _case(lens, 8, 2, 128, seed=21, vmul=ramp)
    _close(_gpu(c), _ref(c), "V scale ramp")


@pytest.mark.parametrize("qmul", [2.0 ** 60, 2.0 ** -60, 1e4])
def test_q_far_outside_fp16_range(qmul):
    """q is brought into fp16 range by a power of two: huge and tiny q give the same result as
    the fp64 oracle (the logit scale divided by the same factor keeps the logits moderate)."""
    c = _case([500, 37], 8, 2, 64, seed=22)
    c["q"] = (c["q"].float() * qmul).to(torch.bfloat16)
    c["scale"] = 0.125 / qmul
    _close(_gpu(c), _ref(c), f"q x {qmul}")


def test_zero_rows_and_deterministic():
    c = _case([400, 250], 16, 4, 128, seed=23)
    c["ks"][c["bt"][0, 3], :, 5] = 0.0           # K row read as zeros: logit 0
    c["kq"][c["bt"][0, 3], :, 5] = 0
    c["vs"][c["bt"][1, 2], :, :] = 0.0           # a whole block of zero V rows
    first = _gpu(c).clone()
    _close(first, _ref(c), "zero rows")
    for _ in range(3):
        assert torch.equal(_gpu(c), first)


def test_llama8b_full_size_sampled_rows():
    wl = W.WORKLOADS["llama8b"]
    lens = W.context_lengths(wl)
    B, hq, hkv, d = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    mb = int((lens.max() + 15) // 16)
    nb = B * mb + 64
    g = torch.Generator(device=DEV).manual_seed(31)
    kq = torch.randint(1, 256, (nb, hkv, 16, d), generator=g, device=DEV, dtype=torch.uint8)
    vq = torch.randint(1, 256, (nb, hkv, 16, d), generator=g, device=DEV, dtype=torch.uint8)
    ks = torch.empty((nb, hkv, 16), device=DEV).exponential_(generator=g) * 0.02
    vs = torch.empty((nb, hkv, 16), device=DEV).exponential_(generator=g) * 0.02
    bt = torch.randperm(nb, device=DEV, generator=g)[: B * mb].view(B, mb).to(torch.int32)
    q = torch.randn((B, hq, d), generator=g, device=DEV).to(torch.bfloat16)
    c = {"q": q, "kq": kq, "ks": ks, "vq": vq, "vs": vs, "bt": bt, "lens": lens.to(DEV), "scale": d ** -0.5}
    err = pkv.new_error_word(DEV)
    out = _gpu(c, err=err)
    assert pkv.read_error(err) == 0
    rng = np.random.default_rng(32)
    rows = sorted({0, B * hq - 1} | set(rng.choice(B * hq, size=40, replace=False).tolist()))
    ref = _ref(c, rows=rows)
    _close(out.view(B * hq, d)[rows], ref, "llama8b INT8 sampled rows")


def test_long_contexts_with_tail_chunks_sampled_rows():
    """Slices long enough for the INT8 partition's tail chunks (about 71 units per worker, so
    one ticket chunk each): sampled rows against the oracle, every ticket taken (the merge
    reports a ticket left over), and the same bits on a second call although the tickets may
    go to other warps."""
    B, hq, hkv, d = 4, 32, 8, 128
    lens = torch.tensor([65536, 65536, 60001, 65521], dtype=torch.int32)
    mb = int((lens.max() + 15) // 16)
    nb = B * mb + 64
    g = torch.Generator(device=DEV).manual_seed(33)
    kq = torch.randint(1, 256, (nb, hkv, 16, d), generator=g, device=DEV, dtype=torch.uint8)
    vq = torch.randint(1, 256, (nb, hkv, 16, d), generator=g, device=DEV, dtype=torch.uint8)
    ks = torch.empty((nb, hkv, 16), device=DEV).exponential_(generator=g) * 0.02
    vs = torch.empty((nb, hkv, 16), device=DEV).exponential_(generator=g) * 0.02
    bt = torch.randperm(nb, device=DEV, generator=g)[: B * mb].view(B, mb).to(torch.int32)
    q = torch.randn((B, hq, d), generator=g, device=DEV).to(torch.bfloat16)
    c = {"q": q, "kq": kq, "ks": ks, "vq": vq, "vs": vs, "bt": bt, "lens": lens.to(DEV), "scale": d ** -0.5}
    err = pkv.new_error_word(DEV)
    out = _gpu(c, err=err)
    assert pkv.read_error(err) == 0
    assert torch.equal(_gpu(c, err=err), out)
    assert pkv.read_error(err) == 0
    rng = np.random.default_rng(34)
    rows = sorted({0, B * hq - 1} | set(rng.choice(B * hq, size=16, replace=False).tolist()))
    ref = _ref(c, rows=rows)
    _close(out.view(B * hq, d)[rows], ref, "long INT8 contexts, sampled rows")


def _slots_at_last(bt, lens):
    return np.array([int(bt[b, (L - 1) // 16]) * 16 + (L - 1) % 16 for b, L in enumerate(lens)], dtype=np.int64)


@pytest.mark.parametrize("d,hq,hkv", [(128, 8, 2), (64, 6, 3), (128, 32, 8)])
@pytest.mark.parametrize("window", [0, 16])
def test_fused_append_q8_equals_append_then_decode(d, hq, hkv, window):
    """paged_decode_attention_append_q8: the pools end as kv_append_q8 leaves them (bit for
    bit, against the oracle), and the output matches the oracle decode over those pools and
    the GPU's own append-then-decode bit for bit."""
    lens = [1, 15, 16, 17, 33, 100, 257]
    c = _case(lens, hq, hkv, d, seed=90 + d + window)
    g = torch.Generator().manual_seed(91)
    k_new = (rand_bf16((len(lens), hkv, d), g) * torch.logspace(-2, 2, len(lens)).view(-1, 1, 1)).to(torch.bfloat16)
    v_new = rand_bf16((len(lens), hkv, d), g)
    k_new[2, 0] = 0.0                                      # a zero row: scale 0, codes 0
    n = lambda t: t.cpu().numpy()
    slots = _slots_at_last(n(c["bt"]), lens)
    ref_pools = oracle.kv_append_q8(n(c["kq"]), n(c["vq"]), n(c["ks"]), n(c["vs"]), bits(k_new), bits(v_new), slots)
    # the same step as two calls, for the bit-identical comparison
    two = {k: c[k].clone() for k in ("kq", "vq", "ks", "vs")}
    pkv.kv_append_q8(two["kq"], two["vq"], two["ks"], two["vs"], k_new.to(DEV), v_new.to(DEV),
                     torch.from_numpy(slots).to(DEV))
    out_two = pkv.paged_decode_attention_q8(c["q"], two["kq"], two["vq"], two["ks"], two["vs"], c["bt"], c["lens"],
                                            c["scale"], window).clone()
    err = pkv.new_error_word(DEV)
    out = pkv.paged_decode_attention_append_q8(c["q"], c["kq"], c["vq"], c["ks"], c["vs"], k_new.to(DEV),
                                               v_new.to(DEV), c["bt"], c["lens"], c["scale"], window, error_word=err)
    torch.cuda.synchronize()
    assert pkv.read_error(err) == 0
    for name, want in zip(("kq", "vq", "ks", "vs"), ref_pools):
        assert np.array_equal(n(c[name]), want), name
    assert torch.equal(out, out_two)
    _close(out, oracle.paged_decode_q8(bits(c["q"]), *[ref_pools[i] for i in (0, 2, 1, 3)], n(c["bt"]),
                                       n(c["lens"]), c["scale"], window), f"fused INT8 append d={d} w={window}")


def test_fused_append_q8_non_finite_row_is_reported_and_skipped():
    lens = [40, 70]
    c = _case(lens, 8, 2, 128, seed=92)
    k_new = torch.ones((2, 2, 128), dtype=torch.bfloat16)
    v_new = torch.ones((2, 2, 128), dtype=torch.bfloat16)
    v_new[1, 1, 7] = float("inf")                          # sequence 1, kv head 1
    before = {k: c[k].clone() for k in ("kq", "vq", "ks", "vs")}
    err = pkv.new_error_word(DEV)
    pkv.paged_decode_attention_append_q8(c["q"], c["kq"], c["vq"], c["ks"], c["vs"], k_new.to(DEV), v_new.to(DEV),
                                         c["bt"], c["lens"], c["scale"], error_word=err)
    torch.cuda.synchronize()
    assert pkv.read_error(err) == pkv.header_constants()["PKV_DEV_BAD_VALUE"]
    blk1, off1 = int(c["bt"][1, 69 // 16]), 69 % 16
    for k in ("kq", "vq", "ks", "vs"):
        assert torch.equal(c[k][blk1, 1, off1], before[k][blk1, 1, off1]), k   # (1, 1): not written
    blk0, off0 = int(c["bt"][0, 39 // 16]), 39 % 16
    # rows of ones: code 127 everywhere (stored as the byte 255)
    assert np.all(code_values(c["kq"][blk0, :, off0]) == 127) and np.all(code_values(c["kq"][blk1, 0, off1]) == 127)


def test_fused_append_q8_llama8b_full_size_sampled_rows():
    wl = W.WORKLOADS["llama8b"]
    lens = W.context_lengths(wl)
    B, hq, hkv, d = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    mb = int((lens.max() + 15) // 16)
    nb = B * mb + 64
    g = torch.Generator(device=DEV).manual_seed(93)
    kq = torch.randint(1, 256, (nb, hkv, 16, d), generator=g, device=DEV, dtype=torch.uint8)
    vq = torch.randint(1, 256, (nb, hkv, 16, d), generator=g, device=DEV, dtype=torch.uint8)
    ks = torch.empty((nb, hkv, 16), device=DEV).exponential_(generator=g) * 0.02
    vs = torch.empty((nb, hkv, 16), device=DEV).exponential_(generator=g) * 0.02
    bt = torch.randperm(nb, device=DEV, generator=g)[: B * mb].view(B, mb).to(torch.int32)
    q = torch.randn((B, hq, d), generator=g, device=DEV).to(torch.bfloat16)
    k_new = torch.randn((B, hkv, d), generator=g, device=DEV).to(torch.bfloat16)
    v_new = torch.randn((B, hkv, d), generator=g, device=DEV).to(torch.bfloat16)
    n = lambda t: t.cpu().numpy()
    slots = _slots_at_last(n(bt), [int(x) for x in lens])
    ref_pools = oracle.kv_append_q8(n(kq), n(vq), n(ks), n(vs), bits(k_new), bits(v_new), slots)
    err = pkv.new_error_word(DEV)
    out = pkv.paged_decode_attention_append_q8(q, kq, vq, ks, vs, k_new, v_new, bt, lens.to(DEV), d ** -0.5,
                                               error_word=err)
    torch.cuda.synchronize()
    assert pkv.read_error(err) == 0
    for name, got, want in zip(("kq", "vq", "ks", "vs"), (kq, vq, ks, vs), ref_pools):
        assert np.array_equal(n(got), want), name
    rng = np.random.default_rng(94)
    rows = sorted({0, B * hq - 1} | set(rng.choice(B * hq, size=40, replace=False).tolist()))
    ref = oracle.paged_decode_q8(bits(q), ref_pools[0], ref_pools[2], ref_pools[1], ref_pools[3], n(bt), n(lens),
                                 d ** -0.5, rows=rows)
    _close(out.view(B * hq, d)[rows], ref, "llama8b fused INT8 append, sampled rows")
