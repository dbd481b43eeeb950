"""Guard bands around every buffer the library writes: each output, workspace and updated pool
is a view into a larger allocation whose bytes before and after it hold a sentinel pattern, and
after the call (which must also succeed and report no device error) the sentinels are intact.
With the memory checker closed on this pool, this is how out-of-bounds writes would show:
a stray store just past a buffer lands in its band.  Each case is small and runs against
inputs built here; results themselves are checked by the parity tests."""
import numpy as np
import pytest
import torch

import paged_kv_cache_mapped_gb300 as pkv
from paged_kv_cache_mapped_gb300 import inputs as W
from helpers import rand_bf16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
BAND = 8192          # bytes of sentinel before and after each buffer (keeps 256-byte alignment)
SENTINEL = 0xA7


class Guarded:
    """A device buffer of `nbytes` (shape/dtype view) between two sentinel bands."""

    def __init__(self, shape, dtype, init=None):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.raw = torch.full((BAND + n + BAND,), SENTINEL, dtype=torch.uint8, device=DEV)
        self.n = n
        self.t = self.raw[BAND:BAND + n].view(dtype).view(shape)
        if isinstance(init, (int, float)):
            self.t.fill_(init)
        elif init is not None:
            self.t.copy_(init)

    def intact(self):
        torch.cuda.synchronize()
        return bool((self.raw[:BAND] == SENTINEL).all()) and bool((self.raw[BAND + self.n:] == SENTINEL).all())


def _check(*bufs):
    for name, b in bufs:
        assert b.intact(), f"{name}: a write landed outside the buffer"


def _layer(lens, hq, hkv, d, seed, nb_extra=6):
    wl = W.Workload("guard", 95, batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    nb = sum((L + 15) // 16 for L in lens) + nb_extra
    return W.make_layer(wl, layer=seed, device=DEV, lengths=lens_t, num_blocks=nb), nb


@pytest.mark.parametrize("d,hq,hkv", [(128, 32, 8), (64, 12, 2)])
def test_decode_out_workspace_and_pools(d, hq, hkv):
    lens = [1, 17, 700, 3000, 0, 256]
    c, nb = _layer(lens, hq, hkv, d, seed=1)
    B = len(lens)
    mb = c["block_tables"].shape[1]
    out = Guarded((B, hq, d), torch.bfloat16)
    ws = Guarded((pkv.decode_workspace_bytes(B, hq, hkv, d, nb, mb),), torch.uint8, init=0)
    kc = Guarded(c["k_cache"].shape, torch.bfloat16, init=c["k_cache"])
    vc = Guarded(c["v_cache"].shape, torch.bfloat16, init=c["v_cache"])
    g = torch.Generator().manual_seed(2)
    k_new = rand_bf16((B, hkv, d), g).to(DEV)
    v_new = rand_bf16((B, hkv, d), g).to(DEV)
    err = pkv.new_error_word(DEV)
    for window in (0, 33):
        pkv.paged_decode_attention(c["q"], kc.t, vc.t, c["block_tables"], c["context_lens"], c["scale"], window,
                                   out=out.t, workspace=ws.t, error_word=err)
        pkv.paged_decode_attention_append(c["q"], kc.t, vc.t, k_new, v_new, c["block_tables"], c["context_lens"],
                                          c["scale"], window, out=out.t, workspace=ws.t, error_word=err,
                                          inputs_ready=True)
    S = mb * 16
    acc = Guarded((B, hkv, S), torch.float32, init=0)
    lse = Guarded((B, hq), torch.float32)
    logits = Guarded((B, hq, S), torch.float32)
    pkv.paged_decode_attention_scores(c["q"], kc.t, vc.t, c["block_tables"], c["context_lens"], c["scale"], acc.t,
                                      out=out.t, lse=lse.t, logits=logits.t, workspace=ws.t, error_word=err)
    assert pkv.read_error(err) == 0
    _check(("out", out), ("workspace", ws), ("k pool", kc), ("v pool", vc), ("scores", acc), ("lse", lse),
           ("logits", logits))


def test_fixed_scratch_out():
    c, nb = _layer([40, 1000, 1], 8, 2, 128, seed=3)
    out = Guarded(c["q"].shape, torch.bfloat16)
    err = pkv.new_error_word(DEV)
    pkv.paged_decode_attention_fixed_scratch(c["q"], c["k_cache"], c["v_cache"], c["block_tables"],
                                             c["context_lens"], c["scale"], out=out.t, error_word=err)
    assert pkv.read_error(err) == 0
    _check(("out", out))


def _q8_pools(nb, hkv, d, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    codes = torch.randint(1, 256, (nb, hkv, 16, d), generator=g, device=DEV, dtype=torch.uint8)
    scales = torch.empty((nb, hkv, 16), device=DEV).exponential_(generator=g) * 0.02
    return codes, scales


def test_int8_append_decode_pools_and_out():
    lens = [5, 300, 2049, 16]
    hq, hkv, d = 16, 4, 128
    c, nb = _layer(lens, hq, hkv, d, seed=4)
    B = len(lens)
    kq0, ks0 = _q8_pools(nb, hkv, d, 5)
    vq0, vs0 = _q8_pools(nb, hkv, d, 6)
    kq = Guarded(kq0.shape, torch.uint8, init=kq0)
    vq = Guarded(vq0.shape, torch.uint8, init=vq0)
    ks = Guarded(ks0.shape, torch.float32, init=ks0)
    vs = Guarded(vs0.shape, torch.float32, init=vs0)
    out = Guarded((B, hq, d), torch.bfloat16)
    ws = Guarded((pkv.decode_workspace_bytes(B, hq, hkv, d, nb, c["block_tables"].shape[1]),), torch.uint8, init=0)
    g = torch.Generator().manual_seed(7)
    k_new = rand_bf16((B, hkv, d), g).to(DEV)
    v_new = rand_bf16((B, hkv, d), g).to(DEV)
    bt = c["block_tables"].cpu()
    slots = torch.tensor([int(bt[b, (L - 1) // 16]) * 16 + (L - 1) % 16 for b, L in enumerate(lens)],
                         dtype=torch.int64, device=DEV)
    err = pkv.new_error_word(DEV)
    pkv.kv_append_q8(kq.t, vq.t, ks.t, vs.t, k_new, v_new, slots, error_word=err)
    pkv.paged_decode_attention_q8(c["q"], kq.t, vq.t, ks.t, vs.t, c["block_tables"], c["context_lens"], c["scale"],
                                  out=out.t, workspace=ws.t, error_word=err)
    pkv.paged_decode_attention_append_q8(c["q"], kq.t, vq.t, ks.t, vs.t, k_new, v_new, c["block_tables"],
                                         c["context_lens"], c["scale"], out=out.t, workspace=ws.t, error_word=err)
    assert pkv.read_error(err) == 0
    _check(("k codes", kq), ("v codes", vq), ("k scales", ks), ("v scales", vs), ("out", out), ("workspace", ws))


def test_sparse_select_compact_gather_and_rolling():
    lens = [3000, 1200, 700]
    hq, hkv, d = 16, 4, 128
    n_sink, n_recent, k_top = 4, 64, 40
    c, nb = _layer(lens, hq, hkv, d, seed=8)
    B = len(lens)
    K = n_sink + n_recent + k_top
    g = torch.Generator().manual_seed(9)
    S = c["block_tables"].shape[1] * 16
    scores = torch.empty((B, hkv, S)).exponential_(generator=g).to(DEV)
    kept = Guarded((B, hkv, K), torch.int32, init=-1)
    kl = Guarded((B,), torch.int32)
    err = pkv.new_error_word(DEV)
    pkv.kv_select_topk(scores, c["context_lens"], n_sink, n_recent, k_top, kept_out=kept.t, kept_lens_out=kl.t,
                       error_word=err)
    dbt, dnb = W.compact_tables(K, B, seed=10)
    dbt = dbt.to(DEV)
    dk = Guarded((dnb, hkv, 16, d), torch.bfloat16, init=0)
    dv = Guarded((dnb, hkv, 16, d), torch.bfloat16, init=0)
    pkv.kv_compact(dk.t, dv.t, dbt, c["k_cache"], c["v_cache"], c["block_tables"], c["context_lens"], kept.t, kl.t,
                   error_word=err)
    out = Guarded((B, hq, d), torch.bfloat16)
    ws = Guarded((pkv.sparse_decode_workspace_bytes(B, hq, hkv, d, nb, c["block_tables"].shape[1], K),),
                 torch.uint8, init=0)
    pkv.sparse_decode_attention(c["q"], c["k_cache"], c["v_cache"], c["block_tables"], c["context_lens"], kept.t,
                                kl.t, c["scale"], out=out.t, workspace=ws.t, error_word=err)
    # INT8 forms of the compaction and the gather decode
    skq, sks = _q8_pools(nb, hkv, d, 11)
    svq, svs = _q8_pools(nb, hkv, d, 12)
    dkq = Guarded((dnb, hkv, 16, d), torch.uint8, init=0)
    dks = Guarded((dnb, hkv, 16), torch.float32, init=0)
    pkv.kv_compact_q8(dkq.t, dkq.t.clone(), dks.t, dks.t.clone(), dbt, skq, svq, sks, svs, c["block_tables"],
                      c["context_lens"], kept.t, kl.t, error_word=err)
    pkv.sparse_decode_attention_q8(c["q"], skq, svq, sks, svs, c["block_tables"], c["context_lens"], kept.t, kl.t,
                                   c["scale"], out=out.t, workspace=ws.t, error_word=err)
    # rolling admission into the compact pool: slot state from the selection
    slot_pos = Guarded((B, hkv, K), torch.int32, init=kept.t)
    slot_score = Guarded((B, hkv, K), torch.float32, init=torch.rand((B, hkv, K), generator=g).to(DEV))
    rkl = Guarded((B,), torch.int32, init=kl.t)
    lens_next = c["context_lens"] + 1
    k_new = rand_bf16((B, hkv, d), g).to(DEV)
    v_new = rand_bf16((B, hkv, d), g).to(DEV)
    pkv.kv_rolling_admit(dk.t, dv.t, dbt, slot_pos.t, slot_score.t, rkl.t, lens_next, k_new, v_new, n_sink,
                         n_recent, error_word=err)
    assert pkv.read_error(err) == 0
    _check(("kept", kept), ("kept_lens", kl), ("compact k", dk), ("compact v", dv), ("out", out), ("workspace", ws),
           ("compact k codes", dkq), ("compact k scales", dks), ("slot_pos", slot_pos), ("slot_score", slot_score),
           ("kept_lens (rolling)", rkl))


def test_prefill_scores_and_lse():
    lens = [600, 100, 1500]
    hq, hkv, d, alpha = 16, 4, 128, 64
    c, nb = _layer(lens, hq, hkv, d, seed=13)
    B = len(lens)
    g = torch.Generator().manual_seed(14)
    q_win = rand_bf16((B, alpha, hq, d), g).to(DEV)
    S = c["block_tables"].shape[1] * 16
    acc = Guarded((B, hkv, S), torch.float32, init=0)
    lse = Guarded((B, hq, alpha), torch.float32)
    err = pkv.new_error_word(DEV)
    pkv.prefill_window_scores(q_win, c["k_cache"], c["block_tables"], c["context_lens"], c["scale"], acc.t,
                              lse=lse.t, error_word=err)
    pkv.prefill_window_scores(q_win, c["k_cache"], c["block_tables"], c["context_lens"], c["scale"], acc.t,
                              lse=lse.t, lse_given=True, error_word=err)
    assert pkv.read_error(err) == 0
    _check(("scores", acc), ("lse", lse))
