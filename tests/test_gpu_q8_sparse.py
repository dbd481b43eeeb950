"""GPU parity of the INT8 sparse-layer path: the score-emitting decode over INT8 pools
(pkv_paged_decode_attention_scores_q8) against oracle.decode_scores_q8, INT8 compaction
(pkv_kv_compact_q8) and INT8 rolling admission (pkv_kv_rolling_admit_q8) bit for bit against
oracle.compact_q8 / oracle.rolling_admit_q8, and the whole layer (append, score, select,
compact, attend) chained on the GPU against the oracle chained on the CPU.

Tolerances: the INT8 logits are fp32 sums of exact fp16 products (codes times q brought into
fp16 range by a power of two) times the row's fp32 scale, relative error ~1e-6 as for bf16
pools, so the score increments and log-sum-exps take the bf16 score test's bounds (relative
5e-4 per increment; lse 1e-4 absolute + 1e-5 relative).  Outputs take the INT8 decode's gate
(max-abs / rel-L2 on outputs divided by max(1, max |ref|)) and are bit-identical to the plain
INT8 decode's."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_mapped_gb300 as pkv
from paged_kv_cache_mapped_gb300 import inputs as W
from helpers import assert_attn_close, bits, code_values, paged_from_contiguous, rand_bf16, stored_codes

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
RTOL, ATOL = 5e-4, 1e-7


def _n(t):
    return t.cpu().numpy()


def _case(lens, hq, hkv, d, seed, kmul=1.0):
    g = torch.Generator().manual_seed(seed)
    B = len(lens)
    lmax = max(max(lens), 1)
    k = rand_bf16((B, lmax, hkv, d), g) * kmul
    v = rand_bf16((B, lmax, hkv, d), g)
    q = rand_bf16((B, hq, d), g)
    nb = sum((L + 15) // 16 for L in lens) + 5
    kc, vc, bt = paged_from_contiguous(k, v, lens, nb, g)
    kq, ks = oracle.quantize_rows(bits(kc))
    vq, vs = oracle.quantize_rows(bits(vc))
    t = lambda a: torch.from_numpy(a).to(DEV)
    return {"q": q.to(DEV), "kq": t(kq), "ks": t(ks), "vq": t(vq), "vs": t(vs), "bt": bt.to(DEV),
            "lens": torch.tensor(lens, dtype=torch.int32, device=DEV), "scale": d ** -0.5}


def _scores_gpu(c, stride, window=0, init=None, err=None, **kw):
    B, hq, d = c["q"].shape
    hkv = c["kq"].shape[1]
    acc = torch.zeros((B, hkv, stride), dtype=torch.float32, device=DEV) if init is None else init.clone()
    before = acc.clone()
    out, lse = pkv.paged_decode_attention_scores_q8(c["q"], c["kq"], c["vq"], c["ks"], c["vs"], c["bt"], c["lens"],
                                                    c["scale"], acc, window, error_word=err, **kw)
    torch.cuda.synchronize()
    return out, lse, (acc - before).double().cpu().numpy()


def _scores_ref(c, stride, window=0, segs=None):
    return oracle.decode_scores_q8(bits(c["q"]), _n(c["kq"]), _n(c["ks"]), _n(c["bt"]), _n(c["lens"]), c["scale"],
                                   window, stride=stride, segs=segs)


def _check_scores(got, ref, what):
    bad = np.abs(got - ref) > RTOL * np.abs(ref) + ATOL
    assert not bad.any(), f"{what}: {bad.sum()} scores off, worst {np.abs(got - ref).max():.3e}"


def _check_lse(got, ref, what):
    ok = np.isclose(got, ref, rtol=1e-5, atol=1e-4) | (np.isneginf(got) & np.isneginf(ref))
    assert ok.all(), f"{what}: lse off by {np.nanmax(np.abs(np.where(np.isfinite(ref), got - ref, 0)))}"


def _close(got, ref, what):
    top = max(1.0, float(np.abs(ref).max()) if ref.size else 1.0)
    assert_attn_close(got.float() / top, ref / top, what)


def _plain_q8(c, window=0):
    out = pkv.paged_decode_attention_q8(c["q"], c["kq"], c["vq"], c["ks"], c["vs"], c["bt"], c["lens"], c["scale"],
                                        window)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("group", [1, 4, 6, 8])
def test_scores_q8_ragged_lengths_all_groups(d, group):
    hkv = 2
    lens = [700, 1, 0, 33, 1500, 16, 257]
    c = _case(lens, hkv * group, hkv, d, seed=d + group, kmul=3.0)
    stride = 1504
    err = pkv.new_error_word(DEV)
    out, lse, delta = _scores_gpu(c, stride, err=err)
    assert pkv.read_error(err) == 0
    ref, ref_lse = _scores_ref(c, stride)
    _check_scores(delta, ref, f"d={d} G={group}")
    _check_lse(_n(lse).astype(np.float64), ref_lse, f"d={d} G={group}")
    expect = np.array([[group if L > 0 else 0] * hkv for L in lens], dtype=np.float64)
    np.testing.assert_allclose(delta.sum(axis=2), expect, rtol=1e-4, atol=1e-6)
    assert torch.equal(out, _plain_q8(c))


@pytest.mark.parametrize("window", [1, 16, 50, 300])
def test_scores_q8_windows_and_existing_scores(window):
    c = _case([900, 70, 301], 16, 4, 128, seed=40 + window)
    stride = 904
    g = torch.Generator().manual_seed(window)
    init = torch.rand((3, 4, stride), generator=g).to(DEV)
    out, lse, delta = _scores_gpu(c, stride, window, init=init)
    ref, ref_lse = _scores_ref(c, stride, window)
    _check_scores(delta, ref, f"window={window}")
    _check_lse(_n(lse).astype(np.float64), ref_lse, f"window={window}")
    assert torch.equal(out, _plain_q8(c, window))


def test_scores_q8_zero_scale_rows():
    c = _case([400, 250], 16, 4, 128, seed=45)
    c["ks"][c["bt"][0, 3], :, 5] = 0.0           # K row read as zeros: logit 0
    c["vs"][c["bt"][1, 2], :, :] = 0.0           # a block of zero V rows
    out, lse, delta = _scores_gpu(c, 400)
    ref, ref_lse = _scores_ref(c, 400)
    _check_scores(delta, ref, "zero rows")
    _check_lse(_n(lse).astype(np.float64), ref_lse, "zero rows")
    n = lambda t: _n(t)
    _close(out, oracle.paged_decode_q8(bits(c["q"]), n(c["kq"]), n(c["ks"]), n(c["vq"]), n(c["vs"]), n(c["bt"]),
                                       n(c["lens"]), c["scale"]), "zero rows output")


def _sample_segs(B, hkv, n, seed):
    rng = np.random.default_rng(seed)
    return sorted({0, B * hkv - 1} | set(rng.choice(B * hkv, size=min(n, B * hkv), replace=False).tolist()))


def test_scores_q8_llama8b_full_size_sampled_segments():
    wl = W.WORKLOADS["llama8b"]
    lens = W.context_lengths(wl)
    B, hq, hkv, d = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    mb = int((lens.max() + 15) // 16)
    nb = B * mb + 64
    g = torch.Generator(device=DEV).manual_seed(41)
    kq = torch.randint(1, 256, (nb, hkv, 16, d), generator=g, device=DEV, dtype=torch.uint8)
    vq = torch.randint(1, 256, (nb, hkv, 16, d), generator=g, device=DEV, dtype=torch.uint8)
    ks = torch.empty((nb, hkv, 16), device=DEV).exponential_(generator=g) * 0.02
    vs = torch.empty((nb, hkv, 16), device=DEV).exponential_(generator=g) * 0.02
    bt = torch.randperm(nb, device=DEV, generator=g)[: B * mb].view(B, mb).to(torch.int32)
    q = torch.randn((B, hq, d), generator=g, device=DEV).to(torch.bfloat16)
    c = {"q": q, "kq": kq, "ks": ks, "vq": vq, "vs": vs, "bt": bt, "lens": lens.to(DEV), "scale": d ** -0.5}
    stride = mb * 16
    err = pkv.new_error_word(DEV)
    out, lse, delta = _scores_gpu(c, stride, err=err)
    assert pkv.read_error(err) == 0
    np.testing.assert_allclose(delta.sum(axis=2), np.full((B, hkv), wl.group), rtol=1e-4)
    segs = _sample_segs(B, hkv, 24, 42)
    ref, ref_lse = _scores_ref(c, stride, segs=segs)
    _check_scores(delta.reshape(-1, stride)[segs], ref, "llama8b INT8")
    G = wl.group
    lse_np = _n(lse).astype(np.float64).reshape(-1)
    got_lse = np.stack([lse_np[(s // hkv) * hq + (s % hkv) * G + np.arange(G)] for s in segs])
    _check_lse(got_lse, ref_lse, "llama8b INT8")
    assert torch.equal(out, _plain_q8(c))


def _q8_pool(nb, hkv, d, seed):
    rng = np.random.default_rng(seed)
    codes = torch.from_numpy(stored_codes(rng.integers(-127, 128, size=(nb, hkv, 16, d))))
    scales = torch.from_numpy(rng.exponential(size=(nb, hkv, 16)).astype(np.float32))
    return codes.to(DEV), scales.to(DEV)


def _compact_case(d, seed, B=4, hkv=4, L=(900, 33, 0, 1500), max_kept=300):
    rng = np.random.default_rng(seed)
    lens = np.array(L, dtype=np.int32)
    smb = int((lens.max() + 15) // 16)
    snb = B * smb + 7
    sk, sks = _q8_pool(snb, hkv, d, seed)
    sv, svs = _q8_pool(snb, hkv, d, seed + 1)
    sbt = rng.permutation(snb)[: B * smb].reshape(B, smb).astype(np.int32)
    kept = np.full((B, hkv, max_kept), -1, dtype=np.int32)
    kl = np.minimum(lens, max_kept).astype(np.int32)
    kl[1] = 17                                                  # a ragged tail block
    for b in range(B):
        for g in range(hkv):
            kept[b, g, :kl[b]] = np.sort(rng.choice(lens[b], size=kl[b], replace=False)) if kl[b] else []
    dmb = (max_kept + 15) // 16
    dnb = B * dmb + 3
    dk, dks = _q8_pool(dnb, hkv, d, seed + 2)
    dv, dvs = _q8_pool(dnb, hkv, d, seed + 3)
    dbt = rng.permutation(dnb)[: B * dmb].reshape(B, dmb).astype(np.int32)
    t = lambda a: torch.from_numpy(a).to(DEV)
    return {"dk": dk, "dv": dv, "dks": dks, "dvs": dvs, "dbt": t(dbt), "sk": sk, "sv": sv, "sks": sks, "svs": svs,
            "sbt": t(sbt), "lens": t(lens), "kept": t(kept), "kl": t(kl)}


def _compact_both(c, err=None):
    ref = oracle.compact_q8(_n(c["dk"]), _n(c["dv"]), _n(c["dks"]), _n(c["dvs"]), _n(c["dbt"]), _n(c["sk"]),
                            _n(c["sv"]), _n(c["sks"]), _n(c["svs"]), _n(c["sbt"]), _n(c["lens"]), _n(c["kept"]),
                            _n(c["kl"]))
    pkv.kv_compact_q8(c["dk"], c["dv"], c["dks"], c["dvs"], c["dbt"], c["sk"], c["sv"], c["sks"], c["svs"], c["sbt"],
                      c["lens"], c["kept"], c["kl"], error_word=err)
    torch.cuda.synchronize()
    return ref


@pytest.mark.parametrize("d", [64, 128])
def test_compact_q8_bit_exact(d):
    c = _compact_case(d, seed=d)
    err = pkv.new_error_word(DEV)
    ref = _compact_both(c, err)
    assert pkv.read_error(err) == 0
    for name, got, want in zip(("k_codes", "v_codes", "k_scales", "v_scales"), (c["dk"], c["dv"], c["dks"], c["dvs"]),
                               ref):
        assert np.array_equal(_n(got), want), name


def test_compact_q8_bad_inputs_are_reported():
    c = _compact_case(64, seed=3)
    c["kept"][1, 2, 4] = 33                                     # L_1 = 33: past the context
    err = pkv.new_error_word(DEV)
    pkv.kv_compact_q8(c["dk"], c["dv"], c["dks"], c["dvs"], c["dbt"], c["sk"], c["sv"], c["sks"], c["svs"], c["sbt"],
                      c["lens"], c["kept"], c["kl"], error_word=err)
    assert pkv.read_error(err, clear=True) == pkv.header_constants()["PKV_DEV_BAD_KEPT_INDEX"]
    c = _compact_case(64, seed=4)
    c["dbt"][0, 1] = 10 ** 6                                    # destination block outside the pool
    pkv.kv_compact_q8(c["dk"], c["dv"], c["dks"], c["dvs"], c["dbt"], c["sk"], c["sv"], c["sks"], c["svs"], c["sbt"],
                      c["lens"], c["kept"], c["kl"], error_word=err)
    assert pkv.read_error(err) == pkv.header_constants()["PKV_DEV_BAD_BLOCK_ID"]


def _rstate(B, hkv, d, cap, seed):
    g = torch.Generator().manual_seed(seed)
    mb = (cap + 15) // 16
    nb = B * mb + 5
    bt = torch.randperm(nb, generator=g)[: B * mb].view(B, mb).to(torch.int32)
    kq, ks = _q8_pool(nb, hkv, d, seed)                         # garbage in unused slots
    vq, vs = _q8_pool(nb, hkv, d, seed + 1)
    return {"kq": kq, "vq": vq, "ks": ks, "vs": vs, "bt": bt.to(DEV),
            "slot_pos": torch.full((B, hkv, cap), -1, dtype=torch.int32, device=DEV),
            "slot_score": torch.zeros((B, hkv, cap), dtype=torch.float32, device=DEV),
            "kept_lens": torch.zeros(B, dtype=torch.int32, device=DEV)}


_RKEYS = ("kq", "vq", "ks", "vs", "slot_pos", "slot_score", "kept_lens")


def _admit_both(st, lens, k_new, v_new, n_sink, n_recent, err=None):
    before = [_n(st[k]) for k in _RKEYS]
    ref = oracle.rolling_admit_q8(before[0], before[1], before[2], before[3], _n(st["bt"]), before[4], before[5],
                                  before[6], _n(lens), bits(k_new), bits(v_new), n_sink, n_recent)
    pkv.kv_rolling_admit_q8(st["kq"], st["vq"], st["ks"], st["vs"], st["bt"], st["slot_pos"], st["slot_score"],
                            st["kept_lens"], lens, k_new, v_new, n_sink, n_recent, error_word=err)
    torch.cuda.synchronize()
    for name, want in zip(_RKEYS, ref):
        assert np.array_equal(_n(st[name]), want), name


@pytest.mark.parametrize("d,k_top", [(64, 24), (128, 24), (128, 23)])  # 60 slots: 16-byte scan; 59: scalar
def test_rolling_admit_q8_steps_bit_exact(d, k_top):
    B, hkv, n_sink, n_recent = 3, 4, 4, 32
    cap = n_sink + k_top + n_recent
    st = _rstate(B, hkv, d, cap, seed=d + k_top)
    g = torch.Generator().manual_seed(d + 2)
    rng = np.random.default_rng(d + k_top)
    err = pkv.new_error_word(DEV)
    for L in range(1, 150):
        lens = torch.full((B,), L, dtype=torch.int32, device=DEV)
        k_new = rand_bf16((B, hkv, d), g) * float(2.0 ** rng.integers(-20, 20))
        _admit_both(st, lens, k_new.to(DEV), rand_bf16((B, hkv, d), g).to(DEV), n_sink, n_recent, err)
        inc = rng.choice([0.0, 0.25, 0.5, 1.0], size=(B, hkv, cap)).astype(np.float32)
        st["slot_score"] += torch.from_numpy(inc).to(DEV)
    assert pkv.read_error(err) == 0
    assert torch.all(st["kept_lens"] == cap)


def test_rolling_admit_q8_non_finite_row_leaves_its_head_unchanged():
    B, hkv, d, cap = 2, 2, 128, 8
    st = _rstate(B, hkv, d, cap, seed=50)
    k_new = torch.ones((B, hkv, d), dtype=torch.bfloat16)
    v_new = torch.ones((B, hkv, d), dtype=torch.bfloat16)
    v_new[1, 0, 3] = float("nan")
    before = [_n(st[k]).copy() for k in _RKEYS]
    err = pkv.new_error_word(DEV)
    pkv.kv_rolling_admit_q8(st["kq"], st["vq"], st["ks"], st["vs"], st["bt"], st["slot_pos"], st["slot_score"],
                            st["kept_lens"], torch.ones(B, dtype=torch.int32, device=DEV), k_new.to(DEV),
                            v_new.to(DEV), 0, 1, error_word=err)
    assert pkv.read_error(err) == pkv.header_constants()["PKV_DEV_BAD_VALUE"]
    blk1 = int(st["bt"][1, 0])
    assert int(st["slot_pos"][1, 0, 0]) == -1                   # (b=1, g=0): nothing written
    assert np.array_equal(_n(st["kq"])[blk1, 0, 0], before[0][blk1, 0, 0])
    assert float(st["ks"][blk1, 0, 0]) == float(before[2][blk1, 0, 0])
    # (1, 1) admitted: a row of ones is code 127 everywhere (stored as the byte 255)
    assert int(st["slot_pos"][1, 1, 0]) == 0 and np.all(code_values(st["kq"][blk1, 1, 0]) == 127)
    blk0 = int(st["bt"][0, 0])
    assert np.all(code_values(st["kq"][blk0, :, 0]) == 127) and torch.all(st["slot_pos"][0, :, 0] == 0)


def test_int8_sparse_layer_chain_matches_the_oracle_chain():
    """One sparse layer over INT8 pools, as a serving step runs it: append the step's token
    (quantized), decode with scores over the full pool for a few steps, select the kept set,
    compact it into the layer's compact pool, then attend over the compact pool.  The GPU
    chain and the oracle chain see the same inputs; each stage's result is compared, and each
    oracle stage takes the GPU's previous output (so a score within tolerance cannot flip the
    selection)."""
    B, hq, hkv, d = 3, 16, 4, 128
    lens0 = [1200, 700, 1500]
    c = _case([L - 1 for L in lens0], hq, hkv, d, seed=60)
    # room for the appended token: one more block per sequence where the last one is full
    g = torch.Generator().manual_seed(61)
    nb = c["kq"].shape[0]
    extra = torch.arange(nb, nb + B, dtype=torch.int32, device=DEV)
    grow = lambda t, n: torch.cat([t, torch.zeros((n,) + t.shape[1:], dtype=t.dtype, device=DEV)])
    for k in ("kq", "vq", "ks", "vs"):
        c[k] = grow(c[k], B)
    mb = c["bt"].shape[1]
    bt = torch.cat([c["bt"], torch.full((B, 1), -1, dtype=torch.int32, device=DEV)], dim=1)
    for b, L in enumerate(lens0):
        if (L - 1) // 16 >= mb or int(bt[b, (L - 1) // 16]) < 0:
            bt[b, (L - 1) // 16] = extra[b]
    c["bt"] = bt
    c["lens"] = torch.tensor(lens0, dtype=torch.int32, device=DEV)
    slots = torch.tensor([int(bt[b, (L - 1) // 16]) * 16 + (L - 1) % 16 for b, L in enumerate(lens0)],
                         dtype=torch.int64, device=DEV)
    k_new = rand_bf16((B, hkv, d), g).to(DEV)
    v_new = rand_bf16((B, hkv, d), g).to(DEV)
    ref_pools = oracle.kv_append_q8(_n(c["kq"]), _n(c["vq"]), _n(c["ks"]), _n(c["vs"]), bits(k_new), bits(v_new),
                                    _n(slots))
    pkv.kv_append_q8(c["kq"], c["vq"], c["ks"], c["vs"], k_new, v_new, slots)
    for name, want in zip(("kq", "vq", "ks", "vs"), ref_pools):
        assert np.array_equal(_n(c[name]), want), name
    stride = 1504
    acc = torch.zeros((B, hkv, stride), dtype=torch.float32, device=DEV)
    ref_acc = np.zeros((B, hkv, stride))
    for _ in range(3):
        c["q"] = rand_bf16((B, hq, d), g).to(DEV)
        pkv.paged_decode_attention_scores_q8(c["q"], c["kq"], c["vq"], c["ks"], c["vs"], c["bt"], c["lens"],
                                             c["scale"], acc)
        ref_acc += _scores_ref(c, stride)[0]
    torch.cuda.synchronize()
    _check_scores(_n(acc).astype(np.float64), ref_acc, "accumulated scores")
    n_sink, n_recent, k_top = 4, 128, 100
    kmax = n_sink + k_top + n_recent
    kept = torch.full((B, hkv, kmax), -1, dtype=torch.int32, device=DEV)
    kl = torch.empty(B, dtype=torch.int32, device=DEV)
    pkv.kv_select_topk(acc, c["lens"], n_sink, n_recent, k_top, kept_out=kept, kept_lens_out=kl)
    ref_kept, ref_kl = oracle.select_topk(_n(acc), _n(c["lens"]), n_sink, n_recent, k_top)
    assert np.array_equal(_n(kl), ref_kl)
    for b in range(B):
        assert np.array_equal(_n(kept)[b, :, :ref_kl[b]], ref_kept[b, :, :ref_kl[b]])
    dmb = (kmax + 15) // 16
    dnb = B * dmb + 2
    dk, dks = _q8_pool(dnb, hkv, d, 62)
    dv, dvs = _q8_pool(dnb, hkv, d, 63)
    dbt = torch.randperm(dnb, generator=g)[: B * dmb].view(B, dmb).to(torch.int32).to(DEV)
    ref_dst = oracle.compact_q8(_n(dk), _n(dv), _n(dks), _n(dvs), _n(dbt), _n(c["kq"]), _n(c["vq"]), _n(c["ks"]),
                                _n(c["vs"]), _n(c["bt"]), _n(c["lens"]), ref_kept, ref_kl)
    pkv.kv_compact_q8(dk, dv, dks, dvs, dbt, c["kq"], c["vq"], c["ks"], c["vs"], c["bt"], c["lens"], kept, kl)
    for name, got, want in zip(("k", "v", "ks", "vs"), (dk, dv, dks, dvs), ref_dst):
        assert np.array_equal(_n(got), want), f"compact {name}"
    out = pkv.paged_decode_attention_q8(c["q"], dk, dv, dks, dvs, dbt, kl, c["scale"])
    torch.cuda.synchronize()
    rk, rv, rks, rvs = ref_dst
    ref_out = oracle.paged_decode_q8(bits(c["q"]), rk, rks, rv, rvs, _n(dbt), ref_kl, c["scale"])
    _close(out, ref_out, "compact INT8 decode")


def test_compact_q8_sparse_workload_full_size_bit_exact():
    """One layer of the sparse workload (16 x 8 heads, 16384-token contexts, Exp(1) scores):
    the GPU selection's kept lists (4 + 512 + 1024) compact INT8 pools into the compact tables,
    bit for bit against the oracle over every row and scale."""
    wl = W.WORKLOADS["sparse"]
    lens = W.context_lengths(wl)
    B, hkv, d, K = wl.batch, wl.num_kv_heads, wl.head_dim, wl.keep_max
    mb = int((lens.max() + 15) // 16)
    snb = B * mb + 16
    g = torch.Generator(device=DEV).manual_seed(71)
    codes = lambda n: torch.randint(1, 256, (n, hkv, 16, d), generator=g, device=DEV, dtype=torch.uint8)
    scales = lambda n: torch.empty((n, hkv, 16), device=DEV).exponential_(generator=g)
    sk, sv, sks, svs = codes(snb), codes(snb), scales(snb), scales(snb)
    sbt = torch.randperm(snb, device=DEV, generator=g)[: B * mb].view(B, mb).to(torch.int32)
    scores = W.make_scores(wl, wl.full_layers, lens, device=DEV, device_rng=True)
    L = lens.to(DEV)
    kept = torch.empty((B, hkv, K), dtype=torch.int32, device=DEV)
    kl = torch.empty((B,), dtype=torch.int32, device=DEV)
    pkv.kv_select_topk(scores, L, wl.n_sink, wl.n_recent, wl.k_top, kept_out=kept, kept_lens_out=kl)
    dbt_cpu, dnb = W.compact_tables(K, B, seed=5)
    dbt = dbt_cpu.to(DEV)
    dk, dv, dks, dvs = codes(dnb), codes(dnb), scales(dnb), scales(dnb)
    ref = oracle.compact_q8(_n(dk), _n(dv), _n(dks), _n(dvs), dbt_cpu.numpy(), _n(sk), _n(sv), _n(sks), _n(svs),
                            _n(sbt), _n(L), _n(kept), _n(kl))
    err = pkv.new_error_word(DEV)
    pkv.kv_compact_q8(dk, dv, dks, dvs, dbt, sk, sv, sks, svs, sbt, L, kept, kl, error_word=err)
    assert pkv.read_error(err) == 0
    for name, got, want in zip(("k_codes", "v_codes", "k_scales", "v_scales"), (dk, dv, dks, dvs), ref):
        assert np.array_equal(_n(got), want), name


def test_rolling_admit_q8_sparse_workload_shape_one_step():
    """16 sequences x 8 kv heads at the full budget of 1540 slots (any slot order): one step's
    admission into INT8 pools, bit for bit against the oracle."""
    B, hkv, d, n_sink, k_top, n_recent = 16, 8, 128, 4, 512, 1024
    cap = n_sink + k_top + n_recent
    L = 16385
    st = _rstate(B, hkv, d, cap, seed=72)
    rng = np.random.default_rng(72)
    scores = rng.exponential(size=(B, hkv, L - 1)).astype(np.float32)
    kept, _ = oracle.select_topk(scores, np.full(B, L - 1, np.int32), n_sink, n_recent, k_top)
    perm = np.stack([np.stack([rng.permutation(cap) for _ in range(hkv)]) for _ in range(B)])
    pos = np.take_along_axis(kept, perm, axis=2).astype(np.int32)
    st["slot_pos"].copy_(torch.from_numpy(pos))
    st["slot_score"].copy_(torch.from_numpy(np.take_along_axis(scores, pos.astype(np.int64), axis=2)))
    st["kept_lens"].fill_(cap)
    g = torch.Generator().manual_seed(73)
    err = pkv.new_error_word(DEV)
    _admit_both(st, torch.full((B,), L, dtype=torch.int32, device=DEV), rand_bf16((B, hkv, d), g).to(DEV),
                rand_bf16((B, hkv, d), g).to(DEV), n_sink, n_recent, err)
    assert pkv.read_error(err) == 0


def _kept_for(lens, hkv, max_kept, seed, kept_lens=None):
    rng = np.random.default_rng(seed)
    B = len(lens)
    kept = np.full((B, hkv, max_kept), -1, dtype=np.int32)
    kl = np.array([min(L, max_kept) for L in lens] if kept_lens is None else kept_lens, dtype=np.int32)
    for b in range(B):
        for g in range(hkv):
            kept[b, g, :kl[b]] = np.sort(rng.choice(lens[b], size=kl[b], replace=False)) if kl[b] else []
    return kept, kl


def _sparse_q8_gpu(c, kept, kl, err=None):
    out = pkv.sparse_decode_attention_q8(c["q"], c["kq"], c["vq"], c["ks"], c["vs"], c["bt"], c["lens"],
                                         torch.from_numpy(kept).to(DEV), torch.from_numpy(kl).to(DEV), c["scale"],
                                         error_word=err)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("group", [1, 4, 8])
def test_sparse_q8_ragged_kept_lists(d, group):
    hkv = 2
    lens = [700, 1, 0, 33, 1500, 16, 257]
    c = _case(lens, hkv * group, hkv, d, seed=100 + d + group, kmul=2.0)
    kept, kl = _kept_for(lens, hkv, 300, seed=d + group, kept_lens=[300, 1, 0, 17, 300, 16, 129])
    err = pkv.new_error_word(DEV)
    out = _sparse_q8_gpu(c, kept, kl, err)
    assert pkv.read_error(err) == 0
    ref = oracle.sparse_decode_q8(bits(c["q"]), _n(c["kq"]), _n(c["ks"]), _n(c["vq"]), _n(c["vs"]), _n(c["bt"]),
                                  _n(c["lens"]), kept, kl, c["scale"])
    _close(out, ref, f"sparse INT8 d={d} G={group}")


def test_sparse_q8_every_token_kept_matches_the_paged_q8_decode():
    lens = [900, 70, 301]
    c = _case(lens, 16, 4, 128, seed=110)
    kept = np.full((3, 4, 900), -1, dtype=np.int32)
    for b, L in enumerate(lens):
        kept[b, :, :L] = np.arange(L)
    out = _sparse_q8_gpu(c, kept, np.array(lens, np.int32))
    ref = oracle.paged_decode_q8(bits(c["q"]), _n(c["kq"]), _n(c["ks"]), _n(c["vq"]), _n(c["vs"]), _n(c["bt"]),
                                 _n(c["lens"]), c["scale"])
    _close(out, ref, "sparse INT8, every token kept")
    _close(_plain_q8(c), ref, "paged INT8")


def test_sparse_q8_bad_kept_index_is_reported():
    lens = [200, 90]
    c = _case(lens, 8, 2, 64, seed=111)
    kept, kl = _kept_for(lens, 2, 64, seed=112)
    kept[1, 1, 5] = 95                                    # past L_1 = 90
    err = pkv.new_error_word(DEV)
    _sparse_q8_gpu(c, kept, kl, err)
    assert pkv.read_error(err) == pkv.header_constants()["PKV_DEV_BAD_KEPT_INDEX"]


def test_sparse_q8_sparse_workload_full_size_sampled_rows():
    """One layer of the sparse workload over INT8 pools (random codes, Exp row scales): the
    GPU selection's kept lists (4 + 512 + 1024 of 16384 tokens) attended by gather."""
    wl = W.WORKLOADS["sparse"]
    lens = W.context_lengths(wl)
    B, hq, hkv, d, K = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.keep_max
    mb = int((lens.max() + 15) // 16)
    nb = B * mb + 16
    g = torch.Generator(device=DEV).manual_seed(113)
    codes = lambda: torch.randint(1, 256, (nb, hkv, 16, d), generator=g, device=DEV, dtype=torch.uint8)
    scales = lambda: torch.empty((nb, hkv, 16), device=DEV).exponential_(generator=g) * 0.02
    c = {"q": torch.randn((B, hq, d), generator=g, device=DEV).to(torch.bfloat16), "kq": codes(), "vq": codes(),
         "ks": scales(), "vs": scales(),
         "bt": torch.randperm(nb, device=DEV, generator=g)[: B * mb].view(B, mb).to(torch.int32),
         "lens": lens.to(DEV), "scale": wl.scale}
    scores = W.make_scores(wl, wl.full_layers, lens, device=DEV, device_rng=True)
    kept = torch.empty((B, hkv, K), dtype=torch.int32, device=DEV)
    kl = torch.empty((B,), dtype=torch.int32, device=DEV)
    pkv.kv_select_topk(scores, c["lens"], wl.n_sink, wl.n_recent, wl.k_top, kept_out=kept, kept_lens_out=kl)
    err = pkv.new_error_word(DEV)
    out = _sparse_q8_gpu(c, _n(kept), _n(kl), err)
    assert pkv.read_error(err) == 0
    rng = np.random.default_rng(114)
    rows = sorted({0, B * hq - 1} | set(rng.choice(B * hq, size=40, replace=False).tolist()))
    ref = oracle.sparse_decode_q8(bits(c["q"]), _n(c["kq"]), _n(c["ks"]), _n(c["vq"]), _n(c["vs"]), _n(c["bt"]),
                                  _n(c["lens"]), _n(kept), _n(kl), c["scale"], rows=rows)
    _close(out.view(B * hq, d)[rows], ref, "sparse workload, INT8 gather")
