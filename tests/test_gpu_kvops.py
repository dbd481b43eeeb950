"""GPU parity of kv_append, kv_select_topk, kv_compact (bit-exact) and sparse_decode_attention
(within the attention tolerance) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_mapped_gb300 as pkv
from paged_kv_cache_mapped_gb300 import inputs as W
from helpers import assert_attn_close, bits, paged_from_contiguous, rand_bf16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
C = pkv.header_constants()


@pytest.mark.parametrize("d", [64, 128])
def test_append_bit_exact_with_skips(d):
    g = torch.Generator().manual_seed(d)
    nb, hkv, T = 37, 4, 50
    kc = rand_bf16((nb, hkv, 16, d), g).to(DEV)
    vc = rand_bf16((nb, hkv, 16, d), g).to(DEV)
    k = rand_bf16((T, hkv, d), g)
    v = rand_bf16((T, hkv, d), g)
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    slots[[3, 11, 40]] = -1
    okc, ovc = oracle.kv_append(bits(kc), bits(vc), bits(k), bits(v), slots.numpy())
    err = pkv.new_error_word(DEV)
    pkv.kv_append(kc, vc, k.to(DEV), v.to(DEV), slots.to(DEV), error_word=err)
    assert pkv.read_error(err) == 0
    assert np.array_equal(bits(kc), okc) and np.array_equal(bits(vc), ovc)


def test_append_bad_slot_is_reported_and_skipped():
    kc = torch.zeros((4, 2, 16, 128), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    k = torch.ones((2, 2, 128), dtype=torch.bfloat16, device=DEV)
    slots = torch.tensor([5, 4 * 16 + 3], dtype=torch.int64, device=DEV)
    err = pkv.new_error_word(DEV)
    pkv.kv_append(kc, vc, k, k, slots, error_word=err)
    assert pkv.read_error(err) == C["PKV_DEV_BAD_SLOT"]
    assert int(torch.count_nonzero(kc)) == 2 * 128          # only the valid token landed


def _topk_both(scores, lens, n_sink, n_recent, k_top):
    okept, okl = oracle.select_topk(scores.numpy(), lens.numpy(), n_sink, n_recent, k_top)
    err = pkv.new_error_word(DEV)
    kept, kl = pkv.kv_select_topk(scores.to(DEV), lens.to(DEV), n_sink, n_recent, k_top, error_word=err)
    assert pkv.read_error(err) == 0
    return okept, okl, kept.cpu().numpy(), kl.cpu().numpy()


def _assert_same_selection(okept, okl, kept, kl):
    assert np.array_equal(okl, kl)
    for b in range(okept.shape[0]):
        n = okl[b]
        assert np.array_equal(okept[b, :, :n], kept[b, :, :n]), b


def test_topk_ragged_ties_and_short_contexts():
    g = torch.Generator().manual_seed(11)
    B, H, S = 6, 4, 3000
    lens = torch.tensor([3000, 10, 60, 61, 1999, 2500], dtype=torch.int32)
    scores = torch.empty((B, H, S)).exponential_(generator=g)
    scores[0, 0, 500:900] = 2.5                     # a wide tie straddling the cut
    scores[1] = torch.round(scores[1] * 4) / 4       # many small ties
    scores[3, :, ::2] = -0.0                         # -0 vs +0 ties
    scores[3, :, 1::2] = 0.0
    scores[4] = -scores[4]                           # negative scores
    _assert_same_selection(*_topk_both(scores, lens, 4, 32, 24))


def test_topk_sparse_workload_layer_bit_exact():
    wl = W.WORKLOADS["sparse"]
    lens = W.context_lengths(wl)
    scores = W.make_scores(wl, 4, lens)
    _assert_same_selection(*_topk_both(scores, lens, wl.n_sink, wl.n_recent, wl.k_top))


def test_topk_nan_reported():
    scores = torch.ones((1, 1, 100))
    scores[0, 0, 50] = float("nan")
    err = pkv.new_error_word(DEV)
    pkv.kv_select_topk(scores.to(DEV), torch.tensor([100], dtype=torch.int32, device=DEV), 2, 4, 8,
                       error_word=err)
    assert pkv.read_error(err) == C["PKV_DEV_BAD_SCORE"]


def _sparse_case(lens, hq, hkv, d, n_keep, seed):
    g = torch.Generator().manual_seed(seed)
    B = len(lens)
    k = rand_bf16((B, max(lens), hkv, d), g)
    v = rand_bf16((B, max(lens), hkv, d), g)
    q = rand_bf16((B, hq, d), g)
    nb = sum((L + 15) // 16 for L in lens) + 3
    kc, vc, bt = paged_from_contiguous(k, v, lens, nb, g, fill=float("nan"))
    rng = np.random.default_rng(seed)
    max_kept = max(n_keep)
    kept = np.full((B, hkv, max_kept), -1, dtype=np.int32)
    for b, L in enumerate(lens):
        for gh in range(hkv):
            kept[b, gh, :n_keep[b]] = np.sort(rng.choice(L, size=n_keep[b], replace=False))
    return dict(q=q, kc=kc, vc=vc, bt=bt, lens=torch.tensor(lens, dtype=torch.int32),
                kept=torch.from_numpy(kept), kl=torch.tensor(n_keep, dtype=torch.int32), scale=d ** -0.5)


@pytest.mark.parametrize("d,hq,hkv", [(128, 32, 8), (128, 12, 2), (64, 8, 8), (128, 8, 1)])
def test_sparse_gather_decode(d, hq, hkv):
    c = _sparse_case([400, 1000, 37, 5], hq, hkv, d, [100, 333, 37, 1], seed=d + hq)
    ref = oracle.sparse_decode(bits(c["q"]), bits(c["kc"]), bits(c["vc"]), c["bt"].numpy(),
                               c["lens"].numpy(), c["kept"].numpy(), c["kl"].numpy(), c["scale"])
    err = pkv.new_error_word(DEV)
    out = pkv.sparse_decode_attention(c["q"].to(DEV), c["kc"].to(DEV), c["vc"].to(DEV), c["bt"].to(DEV),
                                      c["lens"].to(DEV), c["kept"].to(DEV), c["kl"].to(DEV), c["scale"],
                                      error_word=err)
    torch.cuda.synchronize()
    assert pkv.read_error(err) == 0
    assert_attn_close(out, ref, f"sparse gather d={d} hq={hq} hkv={hkv}")


def test_sparse_bad_kept_index_reported():
    c = _sparse_case([100, 50], 4, 2, 128, [20, 10], seed=5)
    c["kept"][1, 0, 3] = 60                       # beyond the context
    err = pkv.new_error_word(DEV)
    out = pkv.sparse_decode_attention(c["q"].to(DEV), c["kc"].to(DEV), c["vc"].to(DEV), c["bt"].to(DEV),
                                      c["lens"].to(DEV), c["kept"].to(DEV), c["kl"].to(DEV), c["scale"],
                                      error_word=err)
    assert pkv.read_error(err) == C["PKV_DEV_BAD_KEPT_INDEX"]
    assert torch.isfinite(out.float()).all()


def test_compact_bit_exact_and_compact_decode_equals_gather():
    c = _sparse_case([300, 1000, 64], 16, 4, 128, [100, 260, 64], seed=9)
    B, hkv = 3, 4
    max_kept = c["kept"].shape[2]
    per_seq = (max_kept + 15) // 16
    dbt, dnb = W.compact_tables(max_kept, B, seed=77)
    dk = torch.zeros((dnb, hkv, 16, 128), dtype=torch.bfloat16)
    dv = torch.zeros_like(dk)
    odk, odv = oracle.compact(bits(dk), bits(dv), dbt.numpy(), bits(c["kc"]), bits(c["vc"]),
                              c["bt"].numpy(), c["lens"].numpy(), c["kept"].numpy(), c["kl"].numpy())
    dk, dv = dk.to(DEV), dv.to(DEV)
    err = pkv.new_error_word(DEV)
    pkv.kv_compact(dk, dv, dbt.to(DEV), c["kc"].to(DEV), c["vc"].to(DEV), c["bt"].to(DEV),
                   c["lens"].to(DEV), c["kept"].to(DEV), c["kl"].to(DEV), error_word=err)
    assert pkv.read_error(err) == 0
    assert np.array_equal(bits(dk), odk) and np.array_equal(bits(dv), odv)
    assert per_seq == dbt.shape[1]
    # paged decode over the compact pool (context = kept count) == sparse gather over the full pool
    q = c["q"].to(DEV)
    comp = pkv.paged_decode_attention(q, dk, dv, dbt.to(DEV), c["kl"].to(DEV), c["scale"])
    gath = pkv.sparse_decode_attention(q, c["kc"].to(DEV), c["vc"].to(DEV), c["bt"].to(DEV),
                                       c["lens"].to(DEV), c["kept"].to(DEV), c["kl"].to(DEV), c["scale"])
    ref = oracle.paged_decode(bits(c["q"]), odk, odv, dbt.numpy(), c["kl"].numpy(), c["scale"])
    assert_attn_close(comp, ref, "compact-pool decode")
    assert_attn_close(gath, ref, "gather decode")


def test_sparse_workload_layer_pipeline():
    """One sparse layer of the layer-wise sparse workload at full size: select -> compact ->
    decode over the compact pool, and gather decode over the full pool; sampled rows vs oracle."""
    wl = W.WORKLOADS["sparse"]
    lens = W.context_lengths(wl)
    case = W.make_layer(wl, layer=4, device=DEV, device_rng=True)
    scores = W.make_scores(wl, 4, lens, device=DEV, device_rng=True)
    err = pkv.new_error_word(DEV)
    kept, kl = pkv.kv_select_topk(scores, case["context_lens"], wl.n_sink, wl.n_recent, wl.k_top,
                                  error_word=err)
    okept, okl = oracle.select_topk(scores.cpu().numpy(), lens.numpy(), wl.n_sink, wl.n_recent, wl.k_top)
    assert np.array_equal(kept.cpu().numpy(), okept) and np.array_equal(kl.cpu().numpy(), okl)
    dbt, dnb = W.compact_tables(wl.keep_max, wl.batch, seed=5)
    dk = torch.empty((dnb, wl.num_kv_heads, 16, wl.head_dim), dtype=torch.bfloat16, device=DEV)
    dv = torch.empty_like(dk)
    dbt = dbt.to(DEV)
    pkv.kv_compact(dk, dv, dbt, case["k_cache"], case["v_cache"], case["block_tables"],
                   case["context_lens"], kept, kl, error_word=err)
    comp = pkv.paged_decode_attention(case["q"], dk, dv, dbt, kl, wl.scale, error_word=err)
    gath = pkv.sparse_decode_attention(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                                       case["context_lens"], kept, kl, wl.scale, error_word=err)
    torch.cuda.synchronize()
    assert pkv.read_error(err) == 0
    rows = sorted({0, 1, 31, 100, 257, 300, 511} | set(range(16 * 32 - 4, 16 * 32)))
    ref = oracle.sparse_decode(bits(case["q"]), bits(case["k_cache"]), bits(case["v_cache"]),
                               case["block_tables"].cpu().numpy(), lens.numpy(), okept, okl,
                               wl.scale, rows=rows)
    idx = torch.tensor(rows, device=DEV)
    assert_attn_close(comp.view(-1, 128)[idx], ref, "sparse layer: compact pool")
    assert_attn_close(gath.view(-1, 128)[idx], ref, "sparse layer: gather")


@pytest.mark.parametrize("k_top", [0, 7, 300])
def test_topk_uncached_long_lists_and_zero_k(k_top):
    """Candidates beyond the shared-memory key cache (n > 40960) and k_top = 0."""
    g = torch.Generator().manual_seed(100 + k_top)
    lens = torch.tensor([60000, 45000, 30000], dtype=torch.int32)
    scores = torch.empty((3, 2, 60000)).exponential_(generator=g)
    scores[0, 1, 1000:9000] = 4.0          # ties across the cut
    _assert_same_selection(*_topk_both(scores, lens, 3, 64, k_top))


@pytest.mark.parametrize("shape", ["uniform_1_2", "block_of_equals", "all_equal", "two_values", "ties_at_cut"])
def test_topk_digit_paths(shape):
    """Score distributions that take each route of the radix select: few keys sharing the first
    12-bit digit (ranked at once), a few thousand sharing it (a short list and a second digit),
    thousands sharing 24 bits (a third digit), and every candidate sharing it (passes over every
    key); bit-exact against the oracle, ties by lower position."""
    g = torch.Generator().manual_seed(77)
    B, H, S = 3, 2, 16384
    lens = torch.tensor([16384, 15000, 9000], dtype=torch.int32)
    if shape == "uniform_1_2":       # one exponent: 8 first-digit bins of ~2000 keys each
        scores = 1.0 + torch.rand((B, H, S), generator=g)
    elif shape == "block_of_equals":  # 2000 equal keys straddling the cut, inside one 24-bit group
        scores = torch.rand((B, H, S), generator=g)
        scores[:, :, 3000:5000] = 0.98765
    elif shape == "all_equal":
        scores = torch.full((B, H, S), 0.5)
    elif shape == "ties_at_cut":      # Exp(1), with 30 more candidates set to the 512th best value
        scores = torch.empty((B, H, S)).exponential_(generator=g)
        for b in range(B):
            L = int(lens[b])
            for h in range(H):
                cand = scores[b, h, 4:L - 1024]
                v = torch.sort(cand, descending=True).values[511]
                below = torch.nonzero(cand < v).flatten()
                pick = below[torch.randperm(below.numel(), generator=g)[:30]]
                cand[pick] = v
    else:                             # two values: the cut falls inside the larger one's ties
        scores = torch.where(torch.rand((B, H, S), generator=g) < 0.02, 2.0, 1.0)
    _assert_same_selection(*_topk_both(scores, lens, 4, 1024, 512))
