"""GPU parity of the rolling admission (pkv_kv_rolling_admit) against the oracle: bit-exact on
the pool, the slot positions, the slot scores and the slot counts, step after step, and in a
loop with the score-emitting decode over the compact pool (the layer's own scores drive which
token is dropped)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_mapped_gb300 as pkv
from helpers import assert_attn_close, bits, rand_bf16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _state(B, hkv, d, cap, seed):
    g = torch.Generator().manual_seed(seed)
    mb = (cap + 15) // 16
    nb = B * mb + 5
    bt = torch.randperm(nb, generator=g)[: B * mb].view(B, mb).to(torch.int32)
    kc = rand_bf16((nb, hkv, 16, d), g)  # garbage in unused slots
    vc = rand_bf16((nb, hkv, 16, d), g)
    return {"k_cache": kc.to(DEV), "v_cache": vc.to(DEV), "block_tables": bt.to(DEV),
            "slot_pos": torch.full((B, hkv, cap), -1, dtype=torch.int32, device=DEV),
            "slot_score": torch.zeros((B, hkv, cap), dtype=torch.float32, device=DEV),
            "kept_lens": torch.zeros(B, dtype=torch.int32, device=DEV)}


def _np(st):
    return (bits(st["k_cache"]), bits(st["v_cache"]), st["slot_pos"].cpu().numpy(),
            st["slot_score"].cpu().numpy(), st["kept_lens"].cpu().numpy())


def _admit_both(st, lens, k_new, v_new, n_sink, n_recent, err=None):
    before = _np(st)
    ref = oracle.rolling_admit(before[0], before[1], st["block_tables"].cpu().numpy(), before[2], before[3],
                               before[4], lens.cpu().numpy(), bits(k_new), bits(v_new), n_sink, n_recent)
    pkv.kv_rolling_admit(st["k_cache"], st["v_cache"], st["block_tables"], st["slot_pos"], st["slot_score"],
                         st["kept_lens"], lens, k_new, v_new, n_sink, n_recent, error_word=err)
    torch.cuda.synchronize()
    got = _np(st)
    for name, a, b in zip(("k_cache", "v_cache", "slot_pos", "slot_score", "kept_lens"), got, ref):
        assert np.array_equal(a, b), name


@pytest.mark.parametrize("d,k_top", [(64, 24), (128, 24), (64, 23)])  # 60 slots: 16-byte scan; 59: scalar
def test_steps_from_empty_to_full_bit_exact(d, k_top):
    B, hkv, n_sink, n_recent = 3, 4, 4, 32
    cap = n_sink + k_top + n_recent
    st = _state(B, hkv, d, cap, seed=d + k_top)
    g = torch.Generator().manual_seed(d + 1)
    rng = np.random.default_rng(d + k_top)
    err = pkv.new_error_word(DEV)
    for L in range(1, 160):
        lens = torch.full((B,), L, dtype=torch.int32, device=DEV)
        _admit_both(st, lens, rand_bf16((B, hkv, d), g).to(DEV), rand_bf16((B, hkv, d), g).to(DEV),
                    n_sink, n_recent, err)
        # this step's attention adds to the slot scores (random stand-in; ties now and then)
        inc = rng.choice([0.0, 0.25, 0.5, 1.0], size=(B, hkv, cap)).astype(np.float32)
        st["slot_score"] += torch.from_numpy(inc).to(DEV)
    assert pkv.read_error(err) == 0
    assert torch.all(st["kept_lens"] == cap)


def test_sparse_workload_shape_one_step():
    """16 sequences x 8 kv heads, 4 sinks + 512 top-k + 1024 recent = 1540 slots, full."""
    B, hkv, d, n_sink, k_top, n_recent = 16, 8, 128, 4, 512, 1024
    cap = n_sink + k_top + n_recent
    L = 16385
    st = _state(B, hkv, d, cap, seed=5)
    rng = np.random.default_rng(5)
    scores = rng.exponential(size=(B, hkv, L - 1)).astype(np.float32)
    kept, kl = oracle.select_topk(scores, np.full(B, L - 1, np.int32), n_sink, n_recent, k_top)
    perm = np.stack([np.stack([rng.permutation(cap) for _ in range(hkv)]) for _ in range(B)])  # any slot order
    pos = np.take_along_axis(kept, perm, axis=2).astype(np.int32)
    st["slot_pos"].copy_(torch.from_numpy(pos))
    st["slot_score"].copy_(torch.from_numpy(np.take_along_axis(scores, pos.astype(np.int64), axis=2)))
    st["kept_lens"].fill_(cap)
    g = torch.Generator().manual_seed(6)
    err = pkv.new_error_word(DEV)
    _admit_both(st, torch.full((B,), L, dtype=torch.int32, device=DEV), rand_bf16((B, hkv, d), g).to(DEV),
                rand_bf16((B, hkv, d), g).to(DEV), n_sink, n_recent, err)
    assert pkv.read_error(err) == 0


def test_invalid_states_are_reported():
    B, hkv, d, n_sink, n_recent = 1, 2, 64, 1, 2
    cap = 6
    st = _state(B, hkv, d, cap, seed=7)
    st["slot_pos"].copy_(torch.tensor([[[0, 5, 1, 9, 10, 11], [0, 5, 1, 9, 4, 11]]], dtype=torch.int32))
    st["slot_score"].copy_(torch.tensor([[[9.0, 0.1, 0.25, 0.25, 0.9, 0.0]] * 2]))
    st["kept_lens"].fill_(cap)
    g = torch.Generator().manual_seed(8)
    err = pkv.new_error_word(DEV)
    before = _np(st)
    pkv.kv_rolling_admit(st["k_cache"], st["v_cache"], st["block_tables"], st["slot_pos"], st["slot_score"],
                         st["kept_lens"], torch.tensor([13], dtype=torch.int32, device=DEV),
                         rand_bf16((1, 2, d), g).to(DEV), rand_bf16((1, 2, d), g).to(DEV), n_sink, n_recent,
                         error_word=err)
    # kv head 1 has no token at the leaving position 10: reported, that head left unchanged
    assert pkv.read_error(err, clear=True) == pkv.header_constants()["PKV_DEV_BAD_KEPT_INDEX"]
    assert np.array_equal(st["slot_pos"][0, 1].cpu().numpy(), before[2][0, 1])
    # kv head 0 is valid: leaving token 10 (0.9) beats the weakest top-k token 5 (0.1), and the
    # new token 12 takes 5's slot
    assert st["slot_pos"][0, 0].cpu().tolist() == [0, 12, 1, 9, 10, 11]
    assert st["slot_score"][0, 0, 1].item() == 0.0
    st["slot_score"][0, 0, 2] = float("nan")
    pkv.kv_rolling_admit(st["k_cache"], st["v_cache"], st["block_tables"], st["slot_pos"], st["slot_score"],
                         st["kept_lens"], torch.tensor([14], dtype=torch.int32, device=DEV),
                         rand_bf16((1, 2, d), g).to(DEV), rand_bf16((1, 2, d), g).to(DEV), n_sink, n_recent,
                         error_word=err)
    code = pkv.read_error(err)
    assert code == pkv.header_constants()["PKV_DEV_BAD_SCORE"]


def test_loop_with_the_layer_own_scores():
    """Each step: admit the token, then attend over the compact pool with the scores going
    straight into the slot scores.  Every admission equals the oracle's on the same state and
    every attention output matches the oracle over the compact pool."""
    B, hkv, hq, d, n_sink, k_top, n_recent = 2, 2, 8, 128, 2, 20, 24
    cap = n_sink + k_top + n_recent
    st = _state(B, hkv, d, cap, seed=9)
    g = torch.Generator().manual_seed(10)
    err = pkv.new_error_word(DEV)
    for L in range(1, 120):
        lens = torch.full((B,), L, dtype=torch.int32, device=DEV)
        _admit_both(st, lens, rand_bf16((B, hkv, d), g).to(DEV), rand_bf16((B, hkv, d), g).to(DEV),
                    n_sink, n_recent, err)
        q = rand_bf16((B, hq, d), g).to(DEV)
        kept = st["kept_lens"].clone()
        out, _ = pkv.paged_decode_attention_scores(q, st["k_cache"], st["v_cache"], st["block_tables"], kept,
                                                   d ** -0.5, st["slot_score"], error_word=err)
        torch.cuda.synchronize()
        if L % 17 == 0:
            ref = oracle.paged_decode(bits(q), bits(st["k_cache"]), bits(st["v_cache"]),
                                      st["block_tables"].cpu().numpy(), kept.cpu().numpy(), d ** -0.5)
            assert_attn_close(out, ref, f"step {L}")
    assert pkv.read_error(err) == 0
