"""Decode calls with PKV_DECODE_INPUTS_READY (the caller declares the pools, block tables and
lengths final before the preceding work on the stream, so the split kernel partitions and starts
its first tile copies before that work ends).

The flag changes when inputs are read, never what is computed: every flagged result is checked
against the fp64 oracle and, bit for bit, against the same call without the flag.  The calls run
back to back on one stream with no synchronisation between them -- the case the flag exists for:
consecutive layers of one decode step, each over its own pools, where a layer's split kernel starts
while the previous layer's kernels finish -- eagerly and captured in a CUDA graph.  The last tests
do the same for kv_select_topk with PKV_SELECT_INPUTS_READY (the scores and lengths final, so the
selection loads and counts them before the preceding work ends) and for kv_compact / kv_compact_q8
with PKV_COMPACT_INPUTS_READY (pools, tables and kept lists final, so the compaction reads the kept
rows before the preceding work ends)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_mapped_gb300 as pkv
from paged_kv_cache_mapped_gb300 import inputs as W
from helpers import assert_attn_close, bits, code_values, paged_from_contiguous, rand_bf16, stored_codes

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _sample_rows(B, hq, n, seed):
    rng = np.random.default_rng(seed)
    rows = {0, B * hq - 1} | {b * hq for b in range(B)}
    rows |= set(rng.choice(B * hq, size=min(n, B * hq), replace=False).tolist())
    return sorted(rows)


def _oracle(case, rows=None, kc=None, vc=None, window=0):
    return oracle.paged_decode(bits(case["q"]), bits(case["k_cache"]) if kc is None else kc,
                               bits(case["v_cache"]) if vc is None else vc, case["block_tables"].cpu().numpy(),
                               case["context_lens"].cpu().numpy(), case["scale"], window, rows=rows)


def _append_call(c, out, ws, ready, err=None, window=0, stream=None):
    return pkv.paged_decode_attention_append(c["q"], c["k_cache"], c["v_cache"], c["k_new"], c["v_new"],
                                             c["block_tables"], c["context_lens"], c["scale"], window, out=out,
                                             workspace=ws, error_word=err, inputs_ready=ready, stream=stream)


def _qwen_layers(layers):
    wl = W.WORKLOADS["qwen1p5b"]
    cases = [W.make_layer(wl, layer=l, device=DEV) for l in layers]
    need = max(pkv.decode_workspace_bytes(wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                          c["num_blocks"], c["max_blocks_per_seq"]) for c in cases)
    return wl, cases, torch.zeros(need, dtype=torch.uint8, device=DEV)


def test_qwen_layer_chain_full_size_against_oracle():
    """Four full-size qwen-shaped layers (0, 1, 2 and 27), each appending this step's token into
    its own pools and attending, issued back to back with the flag: pools bit-exact to the
    oracle's append, sampled rows of every layer within the gate, and every output bit-identical
    to the unflagged calls on the same inputs."""
    wl, cases, ws = _qwen_layers([0, 1, 2, 27])
    pools0 = [(c["k_cache"].clone(), c["v_cache"].clone()) for c in cases]
    err = pkv.new_error_word(DEV)
    outs = [torch.empty_like(c["q"]) for c in cases]
    for c, o in zip(cases, outs):
        _append_call(c, o, ws, True, err)
    torch.cuda.synchronize()
    assert pkv.read_error(err) == 0
    for i, (c, o, (k0, v0)) in enumerate(zip(cases, outs, pools0)):
        okc, ovc = oracle.kv_append(bits(k0), bits(v0), bits(c["k_new"]), bits(c["v_new"]),
                                    c["slot_mapping"].cpu().numpy())
        assert np.array_equal(bits(c["k_cache"]), okc) and np.array_equal(bits(c["v_cache"]), ovc)
        rows = _sample_rows(wl.batch, wl.num_q_heads, 96, 40 + i)
        got = o.view(-1, wl.head_dim)[torch.tensor(rows, device=DEV)]
        assert_attn_close(got, _oracle(c, rows, okc, ovc), f"qwen layer {c['layer']} (flagged)")
    # the same calls without the flag, from the original pools
    for c, (k0, v0), o in zip(cases, pools0, outs):
        c["k_cache"].copy_(k0)
        c["v_cache"].copy_(v0)
        plain = _append_call(c, torch.empty_like(c["q"]), ws, False)
        torch.cuda.synchronize()
        assert torch.equal(plain, o), f"layer {c['layer']}: flagged and plain results differ"


def _small(lens, hq, hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    B, lmax = len(lens), max(max(lens), 1)
    k, v = rand_bf16((B, lmax, hkv, d), g), rand_bf16((B, lmax, hkv, d), g)
    nb = sum((L + 15) // 16 for L in lens) + 3
    kc, vc, bt = paged_from_contiguous(k, v, lens, nb, g, fill=float("nan"))
    case = {"q": rand_bf16((B, hq, d), g).to(DEV), "k_cache": kc.to(DEV), "v_cache": vc.to(DEV),
            "block_tables": bt.to(DEV), "context_lens": torch.tensor(lens, dtype=torch.int32, device=DEV),
            "scale": d ** -0.5, "k_new": rand_bf16((B, hkv, d), g).to(DEV),
            "v_new": rand_bf16((B, hkv, d), g).to(DEV)}
    bt = case["block_tables"].cpu()
    case["slot_mapping"] = torch.tensor([int(bt[b, (L - 1) // 16]) * 16 + (L - 1) % 16 if L > 0 else -1
                                         for b, L in enumerate(lens)], dtype=torch.int64)
    return case


@pytest.mark.parametrize("window", [0, 1, 50])
def test_ragged_shapes_back_to_back(window):
    """Ragged batches of several shapes (d 64 and 128, G 1-8, empty and one-token sequences),
    plain and fused-append calls alternating, all flagged and sharing one workspace, with no
    synchronisation between them; every element against the oracle and bit-identical to the
    unflagged calls."""
    shapes = [([1, 15, 16, 17, 33, 100, 257], 8, 2, 128), ([0, 700, 33], 16, 2, 64),
              ([4000, 1, 2500, 17], 32, 8, 128), ([90] * 12, 8, 8, 64), ([3, 1500], 48, 6, 128)]
    cases = [_small(l, hq, hkv, d, 300 + i) for i, (l, hq, hkv, d) in enumerate(shapes)]
    need = max(pkv.decode_workspace_bytes(c["q"].shape[0], c["q"].shape[1], c["k_cache"].shape[1],
                                          c["k_cache"].shape[3], c["k_cache"].shape[0], c["block_tables"].shape[1])
               for c in cases)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    pools0 = [(c["k_cache"].clone(), c["v_cache"].clone()) for c in cases]

    def run(ready):
        outs = []
        for i, c in enumerate(cases):
            o = torch.empty_like(c["q"])
            if i % 2 == 0 and int(c["context_lens"].min()) > 0:
                _append_call(c, o, ws, ready, err, window)
            else:
                pkv.paged_decode_attention(c["q"], c["k_cache"], c["v_cache"], c["block_tables"],
                                           c["context_lens"], c["scale"], window, out=o, workspace=ws,
                                           error_word=err, inputs_ready=ready)
            outs.append(o)
        return outs

    err = pkv.new_error_word(DEV)
    flagged = run(True)
    torch.cuda.synchronize()
    assert pkv.read_error(err) == 0
    for i, (c, o, (k0, v0)) in enumerate(zip(cases, flagged, pools0)):
        appended = i % 2 == 0 and int(c["context_lens"].min()) > 0
        if appended:
            okc, ovc = oracle.kv_append(bits(k0), bits(v0), bits(c["k_new"]), bits(c["v_new"]),
                                        c["slot_mapping"].numpy())
            assert np.array_equal(bits(c["k_cache"]), okc) and np.array_equal(bits(c["v_cache"]), ovc)
            ref = _oracle(c, None, okc, ovc, window)
        else:
            ref = _oracle(c, None, window=window)
        assert_attn_close(o, ref, f"shape {i} window {window} (flagged)")
    for c, (k0, v0) in zip(cases, pools0):
        c["k_cache"].copy_(k0)
        c["v_cache"].copy_(v0)
    plain = run(False)
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(flagged, plain)):
        assert torch.equal(a, b), f"shape {i}: flagged and plain results differ"


def test_next_query_from_previous_output():
    """The flag lets the split kernel start before the preceding kernel ends, but q is read only
    after it: a call whose q is the previous flagged call's output (written by that call's merge
    and split kernels) gives the result of the same call made after a synchronisation."""
    c1 = _small([2000, 37, 900, 4000], 16, 4, 128, 401)
    c2 = _small([1200, 3000, 16, 64], 16, 4, 128, 402)
    ws = torch.zeros(pkv.decode_workspace_bytes(4, 16, 4, 128, max(c1["k_cache"].shape[0], c2["k_cache"].shape[0]),
                                                max(c1["block_tables"].shape[1], c2["block_tables"].shape[1])),
                     dtype=torch.uint8, device=DEV)
    mid = torch.empty_like(c1["q"])
    out = torch.empty_like(c2["q"])
    for _ in range(3):
        mid.fill_(float("nan"))
        pkv.paged_decode_attention(c1["q"], c1["k_cache"], c1["v_cache"], c1["block_tables"], c1["context_lens"],
                                   c1["scale"], out=mid, workspace=ws, inputs_ready=True)
        pkv.paged_decode_attention(mid, c2["k_cache"], c2["v_cache"], c2["block_tables"], c2["context_lens"],
                                   c2["scale"], out=out, workspace=ws, inputs_ready=True)
        torch.cuda.synchronize()
        assert_attn_close(mid, _oracle(c1), "first call")
        ref = pkv.paged_decode_attention(mid.clone(), c2["k_cache"], c2["v_cache"], c2["block_tables"],
                                         c2["context_lens"], c2["scale"], workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)


def test_graph_of_flagged_layers_matches_eager_plain():
    """Four qwen-shaped layers (fused append + decode, the flag set) captured in one CUDA graph and
    replayed: every layer's output equals the eager unflagged call's bit for bit, and the pools
    hold the appended rows."""
    wl, cases, ws = _qwen_layers([3, 4, 5, 6])
    pools0 = [(c["k_cache"].clone(), c["v_cache"].clone()) for c in cases]
    eager = [_append_call(c, torch.empty_like(c["q"]), ws, False).clone() for c in cases]
    torch.cuda.synchronize()
    appended = [(c["k_cache"].clone(), c["v_cache"].clone()) for c in cases]
    outs = [torch.empty_like(c["q"]) for c in cases]
    s = torch.cuda.Stream(DEV)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        for c, o in zip(cases, outs):   # warm-up on the capture stream
            _append_call(c, o, ws, True)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=s):
            for c, o in zip(cases, outs):
                _append_call(c, o, ws, True, stream=s)
    for _ in range(2):
        for c, (k0, v0) in zip(cases, pools0):
            c["k_cache"].copy_(k0)
            c["v_cache"].copy_(v0)
        for o in outs:
            o.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        for i, (c, o, e, (ka, va)) in enumerate(zip(cases, outs, eager, appended)):
            assert torch.equal(o, e), f"layer {i}"
            assert torch.equal(c["k_cache"], ka) and torch.equal(c["v_cache"], va)


def test_large_batch_record_written_after_wait():
    """Batches above 256 sequences hand the merge a record of unit starts in the workspace; with
    the flag it is written after the preceding kernel ends.  Two different 320-sequence layers
    back to back share the workspace."""
    cases = []
    for layer in range(2):
        wl = W.Workload("batch320", 91, batch=320, num_q_heads=8, num_kv_heads=2, head_dim=128,
                        len_uniform=(0, 3000))
        lens = W.context_lengths(wl)
        lens[layer::37] = 0
        cases.append(W.make_layer(wl, layer=layer, device=DEV, lengths=lens, device_rng=True))
    need = max(pkv.decode_workspace_bytes(320, 8, 2, 128, c["num_blocks"], c["max_blocks_per_seq"]) for c in cases)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    err = pkv.new_error_word(DEV)
    outs = [pkv.paged_decode_attention(c["q"], c["k_cache"], c["v_cache"], c["block_tables"], c["context_lens"],
                                       c["scale"], workspace=ws, error_word=err, inputs_ready=True) for c in cases]
    torch.cuda.synchronize()
    assert pkv.read_error(err) == 0
    for i, (c, o) in enumerate(zip(cases, outs)):
        rows = _sample_rows(320, 8, 120, 60 + i)
        assert_attn_close(o.view(-1, 128)[torch.tensor(rows, device=DEV)], _oracle(c, rows), f"batch 320 layer {i}")
        plain = pkv.paged_decode_attention(c["q"], c["k_cache"], c["v_cache"], c["block_tables"],
                                           c["context_lens"], c["scale"], workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(plain, o)


def test_errors_found_before_the_wait_are_recorded():
    """A bad block id met while the first tiles are issued (before the wait) and a bad context
    length met by the partition are still recorded, once the preceding kernel has ended."""
    codes = pkv.header_constants()
    c = _small([100, 40], 8, 2, 128, 501)
    c["block_tables"][1, 0] = c["k_cache"].shape[0] + 5
    err = pkv.new_error_word(DEV)
    pkv.paged_decode_attention(c["q"], c["k_cache"], c["v_cache"], c["block_tables"], c["context_lens"],
                               c["scale"], error_word=err, inputs_ready=True)
    assert pkv.read_error(err) == codes["PKV_DEV_BAD_BLOCK_ID"]
    c2 = _small([100, 40], 8, 2, 128, 502)
    c2["context_lens"][0] = 16 * c2["block_tables"].shape[1] + 1
    err2 = pkv.new_error_word(DEV)
    out = pkv.paged_decode_attention(c2["q"], c2["k_cache"], c2["v_cache"], c2["block_tables"],
                                     c2["context_lens"], c2["scale"], error_word=err2, inputs_ready=True)
    assert pkv.read_error(err2) == codes["PKV_DEV_BAD_CONTEXT_LEN"]
    ref = _oracle({**c2, "q": c2["q"][1:], "block_tables": c2["block_tables"][1:],
                   "context_lens": c2["context_lens"][1:]})
    assert_attn_close(out[1:], ref, "valid sequence beside a bad length")


def _q8_pools(nb, hkv, d, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    codes = lambda: torch.randint(1, 256, (nb, hkv, 16, d), generator=g, device=DEV, dtype=torch.uint8)
    scales = lambda: torch.empty((nb, hkv, 16), device=DEV).exponential_(generator=g) * 0.02
    return codes(), codes(), scales(), scales()


def test_int8_scores_and_sparse_forms_flagged_equal_plain():
    """The INT8 fused append, the score-emitting decode and the gather form of the sparse decode
    take the flag too: back to back, their results equal the unflagged calls' bit for bit."""
    wl, cases, ws = _qwen_layers([7, 8])
    hkv, d = wl.num_kv_heads, wl.head_dim
    p8 = [_q8_pools(c["num_blocks"], hkv, d, 70 + i) for i, c in enumerate(cases)]
    p80 = [tuple(t.clone() for t in p) for p in p8]

    def q8(ready):
        outs = []
        for c, p in zip(cases, p8):
            outs.append(pkv.paged_decode_attention_append_q8(
                c["q"], *p, c["k_new"], c["v_new"], c["block_tables"], c["context_lens"], c["scale"], workspace=ws,
                inputs_ready=ready))
        torch.cuda.synchronize()
        return outs
    a = q8(True)
    after = [tuple(t.clone() for t in p) for p in p8]
    for p, p0 in zip(p8, p80):
        for t, t0 in zip(p, p0):
            t.copy_(t0)
    b = q8(False)
    for i in range(2):
        assert torch.equal(a[i], b[i]), f"INT8 layer {i}"
        assert all(torch.equal(x, y) for x, y in zip(after[i], p8[i]))

    S = cases[0]["block_tables"].shape[1] * 16

    def scores(ready):
        res = []
        for c in cases:
            acc = torch.zeros((wl.batch, hkv, S), dtype=torch.float32, device=DEV)
            o, lse = pkv.paged_decode_attention_scores(c["q"], c["k_cache"], c["v_cache"], c["block_tables"],
                                                       c["context_lens"], c["scale"], acc, workspace=ws,
                                                       inputs_ready=ready)
            res.append((o, lse, acc))
        torch.cuda.synchronize()
        return res
    for (o1, l1, s1), (o2, l2, s2) in zip(scores(True), scores(False)):
        assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(s1, s2)

    # gather form: kept lists of sinks, a strided middle and the recent window
    def kept_for(c):
        lens = c["context_lens"].cpu()
        mk = 4 + 64 + 256
        kept = torch.zeros((wl.batch, hkv, mk), dtype=torch.int32)
        klen = torch.zeros(wl.batch, dtype=torch.int32)
        for bb in range(wl.batch):
            L = int(lens[bb])
            if L <= mk:
                lst = list(range(L))
            else:
                mid = list(range(4, L - 256, max(1, (L - 260) // 64)))[:64]
                lst = sorted(set(range(4)) | set(mid) | set(range(L - 256, L)))
            klen[bb] = len(lst)
            kept[bb, :, :len(lst)] = torch.tensor(lst, dtype=torch.int32)
        return kept.to(DEV), klen.to(DEV)
    kls = [kept_for(c) for c in cases]

    def sparse(ready):
        outs = [pkv.sparse_decode_attention(c["q"], c["k_cache"], c["v_cache"], c["block_tables"], c["context_lens"],
                                            kl[0], kl[1], c["scale"], workspace=ws, inputs_ready=ready)
                for c, kl in zip(cases, kls)]
        torch.cuda.synchronize()
        return outs
    for i, (x, y) in enumerate(zip(sparse(True), sparse(False))):
        assert torch.equal(x, y), f"sparse layer {i}"
        c, (kept, klen) = cases[i], kls[i]
        rows = _sample_rows(wl.batch, wl.num_q_heads, 48, 80 + i)
        ref = oracle.sparse_decode(bits(c["q"]), bits(c["k_cache"]), bits(c["v_cache"]),
                                   c["block_tables"].cpu().numpy(), c["context_lens"].cpu().numpy(),
                                   kept.cpu().numpy(), klen.cpu().numpy(), c["scale"], rows=rows)
        assert_attn_close(x.view(-1, d)[torch.tensor(rows, device=DEV)], ref, f"sparse layer {i} (flagged)")


# ---------------------------------------------------------------- kv_select_topk with the flag

def test_select_layers_back_to_back_against_oracle():
    """PKV_SELECT_INPUTS_READY: the selections of several layers, each from its own final scores
    (Exp(1), ties, ragged lengths, short lists), run back to back on one stream with no
    synchronisation, writing into one shared pair of output buffers after each layer's copy;
    every layer's kept lists equal the oracle's and the unflagged call's, bit for bit."""
    g = torch.Generator().manual_seed(71)
    B, hkv, S = 5, 3, 6000
    lens = torch.tensor([6000, 5000, 40, 0, 3333], dtype=torch.int32)
    n_sink, n_recent, k_top = 3, 64, 300
    layers = [torch.empty((B, hkv, S)).exponential_(generator=g) for _ in range(3)]
    layers.append(torch.round(torch.empty((B, hkv, S)).exponential_(generator=g) * 4) / 4)  # ties
    dl = lens.to(DEV)
    kmax = n_sink + k_top + n_recent
    kept = torch.empty((B, hkv, kmax), dtype=torch.int32, device=DEV)
    kl = torch.empty(B, dtype=torch.int32, device=DEV)
    err = pkv.new_error_word(DEV)
    got = []
    for sc in layers:
        pkv.kv_select_topk(sc.to(DEV), dl, n_sink, n_recent, k_top, kept_out=kept, kept_lens_out=kl,
                           error_word=err, inputs_ready=True)
        got.append((kept.clone(), kl.clone()))  # the copies queue behind the flagged call
    torch.cuda.synchronize()
    assert pkv.read_error(err) == 0
    for sc, (k, n) in zip(layers, got):
        okept, okl = oracle.select_topk(sc.numpy(), lens.numpy(), n_sink, n_recent, k_top)
        assert np.array_equal(n.cpu().numpy(), okl)
        kc = k.cpu().numpy()
        for b in range(B):
            assert np.array_equal(kc[b, :, :okl[b]], okept[b, :, :okl[b]])
        pk, pl = pkv.kv_select_topk(sc.to(DEV), dl, n_sink, n_recent, k_top)
        torch.cuda.synchronize()
        assert torch.equal(pl, n)
        for b in range(B):
            assert torch.equal(pk[b, :, :int(okl[b])], k[b, :, :int(okl[b])])


def test_select_flagged_in_graph_and_errors_after_the_wait():
    """Flagged selections captured in a CUDA graph equal the eager unflagged ones; a length out of
    range found before the wait is recorded once the call may write (PKV_DEV_BAD_CONTEXT_LEN)."""
    g = torch.Generator().manual_seed(72)
    B, hkv, S = 4, 2, 3000
    lens = torch.tensor([3000, 2999, 700, 1], dtype=torch.int32, device=DEV)
    scores = [torch.empty((B, hkv, S)).exponential_(generator=g).to(DEV) for _ in range(4)]
    outs = [(torch.empty((B, hkv, 4 + 50 + 200), dtype=torch.int32, device=DEV),
             torch.empty(B, dtype=torch.int32, device=DEV)) for _ in scores]
    s = torch.cuda.Stream(DEV)
    with torch.cuda.stream(s):
        pkv.kv_select_topk(scores[0], lens, 4, 200, 50, stream=s)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            for sc, (k, n) in zip(scores, outs):
                pkv.kv_select_topk(sc, lens, 4, 200, 50, kept_out=k, kept_lens_out=n, inputs_ready=True, stream=s)
        gr.replay()
        torch.cuda.synchronize()
    for sc, (k, n) in zip(scores, outs):
        pk, pl = pkv.kv_select_topk(sc, lens, 4, 200, 50)
        torch.cuda.synchronize()
        assert torch.equal(pl, n)
        for b in range(B):
            assert torch.equal(pk[b, :, :int(pl[b])], k[b, :, :int(pl[b])])
    err = pkv.new_error_word(DEV)
    bad = torch.tensor([3000, S + 1, 700, 1], dtype=torch.int32, device=DEV)
    pkv.kv_select_topk(scores[1], bad, 4, 200, 50, error_word=err, inputs_ready=True)
    torch.cuda.synchronize()
    assert pkv.read_error(err) == pkv.header_constants()["PKV_DEV_BAD_CONTEXT_LEN"]


@pytest.mark.parametrize("S", [16387, 50003])
def test_select_flagged_long_and_odd_rows(S):
    """Flagged selections over rows that fill the key cache (a row length that is not a multiple
    of 4: the cache rounds up and the loads are unaligned) and rows longer than the cache (the
    general path reads the scores again), each against the oracle and the unflagged call."""
    g = torch.Generator().manual_seed(73 + S)
    B, hkv = 3, 2
    lens = torch.tensor([S, S - 5, 9000], dtype=torch.int32)
    n_sink, n_recent, k_top = 4, 128, 700
    layers = [torch.empty((B, hkv, S)).exponential_(generator=g) for _ in range(2)]
    err = pkv.new_error_word(DEV)
    got = [pkv.kv_select_topk(sc.to(DEV), lens.to(DEV), n_sink, n_recent, k_top, error_word=err, inputs_ready=True)
           for sc in layers]
    torch.cuda.synchronize()
    assert pkv.read_error(err) == 0
    for sc, (k, n) in zip(layers, got):
        okept, okl = oracle.select_topk(sc.numpy(), lens.numpy(), n_sink, n_recent, k_top)
        assert np.array_equal(n.cpu().numpy(), okl)
        pk, _ = pkv.kv_select_topk(sc.to(DEV), lens.to(DEV), n_sink, n_recent, k_top)
        torch.cuda.synchronize()
        kc, pc = k.cpu().numpy(), pk.cpu().numpy()
        for b in range(B):
            assert np.array_equal(kc[b, :, :okl[b]], okept[b, :, :okl[b]])
            assert np.array_equal(pc[b, :, :okl[b]], kc[b, :, :okl[b]])


def _compact_layer(B, hkv, d, lens, max_kept, seed, q8):
    """One layer's source pool (bf16, or INT8 codes with Exp row scales), its shuffled block table
    and strictly rising kept lists (min(L_b, max_kept) tokens, one list a ragged 17)."""
    rng = np.random.default_rng(seed)
    lens = np.array(lens, dtype=np.int32)
    smb = int((lens.max() + 15) // 16)
    snb = B * smb + 5
    sbt = rng.permutation(snb)[: B * smb].reshape(B, smb).astype(np.int32)
    kl = np.minimum(lens, max_kept).astype(np.int32)
    kl[1] = min(17, lens[1])
    kept = np.full((B, hkv, max_kept), -1, dtype=np.int32)
    for b in range(B):
        for g in range(hkv):
            if kl[b]:
                kept[b, g, :kl[b]] = np.sort(rng.choice(lens[b], size=kl[b], replace=False))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    c = {"sbt": t(sbt), "lens": t(lens), "kept": t(kept), "kl": t(kl)}
    if q8:
        for name in ("sk", "sv"):
            c[name] = t(stored_codes(rng.integers(-127, 128, size=(snb, hkv, 16, d))))
            c[name + "s"] = t(rng.exponential(size=(snb, hkv, 16)).astype(np.float32))
    else:
        for name in ("sk", "sv"):
            c[name] = t(rng.integers(0, 1 << 16, size=(snb, hkv, 16, d)).astype(np.uint16)).view(torch.bfloat16)
    return c


def _compact_dst(B, hkv, d, max_kept, seed, q8):
    """A destination pool filled with noise (slots the copy does not address keep it) and its table."""
    rng = np.random.default_rng(seed)
    dmb = (max_kept + 15) // 16
    dnb = B * dmb + 3
    dbt = torch.from_numpy(rng.permutation(dnb)[: B * dmb].reshape(B, dmb).astype(np.int32)).to(DEV)
    if q8:
        pools = [torch.from_numpy(stored_codes(rng.integers(-127, 128, size=(dnb, hkv, 16, d)))).to(DEV)
                 for _ in range(2)]
        pools += [torch.from_numpy(rng.exponential(size=(dnb, hkv, 16)).astype(np.float32)).to(DEV) for _ in range(2)]
    else:
        pools = [torch.from_numpy(rng.integers(0, 1 << 16, size=(dnb, hkv, 16, d)).astype(np.uint16)).to(DEV)
                 .view(torch.bfloat16) for _ in range(2)]
    return pools, dbt


def _compact_call(c, pools, dbt, q8, ready, err=None, stream=None):
    if q8:
        pkv.kv_compact_q8(pools[0], pools[1], pools[2], pools[3], dbt, c["sk"], c["sv"], c["sks"], c["svs"],
                          c["sbt"], c["lens"], c["kept"], c["kl"], error_word=err, inputs_ready=ready, stream=stream)
    else:
        pkv.kv_compact(pools[0], pools[1], dbt, c["sk"], c["sv"], c["sbt"], c["lens"], c["kept"], c["kl"],
                       error_word=err, inputs_ready=ready, stream=stream)


def _np(t):
    return (t.view(torch.uint16) if t.dtype == torch.bfloat16 else t).cpu().numpy()


def _compact_oracle(c, pools, dbt, q8):
    """The destination pools after one compaction, by the oracle (numpy copies of `pools`)."""
    n = lambda k: _np(c[k])
    if q8:
        return list(oracle.compact_q8(*pools, _np(dbt), n("sk"), n("sv"), n("sks"), n("svs"), n("sbt"), n("lens"),
                                      n("kept"), n("kl")))
    return list(oracle.compact(*pools, _np(dbt), n("sk"), n("sv"), n("sbt"), n("lens"), n("kept"), n("kl")))


@pytest.mark.parametrize("q8,d", [(False, 128), (False, 64), (True, 128), (True, 64)])
def test_compact_layers_back_to_back_against_oracle(q8, d):
    """PKV_COMPACT_INPUTS_READY: the compactions of several layers, each from its own pool through
    final kept lists, run back to back into one shared destination pool with a copy of that pool
    queued after each (the next flagged call may read before the copy ends and must write after
    it); every copy equals the oracle's chain of compactions and the unflagged chain, bit for bit."""
    B, hkv, max_kept = 4, 3, 300
    layers = [_compact_layer(B, hkv, d, [900, 33, 0, 1500], max_kept, 80 + l, q8) for l in range(3)]
    pools, dbt = _compact_dst(B, hkv, d, max_kept, 90, q8)
    start = [p.clone() for p in pools]
    err = pkv.new_error_word(DEV)
    torch.cuda.synchronize()
    snaps = []
    for c in layers:
        _compact_call(c, pools, dbt, q8, True, err)
        snaps.append([p.clone() for p in pools])
    torch.cuda.synchronize()
    assert pkv.read_error(err) == 0
    want = [_np(p) for p in start]
    for c, snap in zip(layers, snaps):
        want = _compact_oracle(c, want, dbt, q8)
        for w, g in zip(want, snap):
            assert np.array_equal(_np(g), w)
    plain = [p.clone() for p in start]
    for c, snap in zip(layers, snaps):
        _compact_call(c, plain, dbt, q8, False)
        torch.cuda.synchronize()
        for p, g in zip(plain, snap):
            assert torch.equal(_np_t(p), _np_t(g))


def _np_t(t):
    return t.view(torch.uint16) if t.dtype == torch.bfloat16 else t


@pytest.mark.parametrize("q8", [False, True])
def test_compact_flagged_in_graph_and_errors_after_the_wait(q8):
    """Flagged compactions of four layers into four pools, captured in a CUDA graph, equal the eager
    unflagged ones; a kept entry past its context, a source block id and a destination block id
    outside their pools, found before the wait, are recorded once the call may write."""
    B, hkv, d, max_kept = 3, 2, 128, 200
    layers = [_compact_layer(B, hkv, d, [700, 40, 2000], max_kept, 100 + l, q8) for l in range(4)]
    dsts = [_compact_dst(B, hkv, d, max_kept, 110 + l, q8) for l in range(4)]
    start = [[p.clone() for p in pools] for pools, _ in dsts]
    s = torch.cuda.Stream(DEV)
    with torch.cuda.stream(s):
        _compact_call(layers[0], [p.clone() for p in start[0]], dsts[0][1], q8, False, stream=s)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            for c, (pools, dbt) in zip(layers, dsts):
                _compact_call(c, pools, dbt, q8, True, stream=s)
        gr.replay()
        torch.cuda.synchronize()
    for c, (pools, dbt), st in zip(layers, dsts, start):
        _compact_call(c, st, dbt, q8, False)
        torch.cuda.synchronize()
        for p, g in zip(st, pools):
            assert torch.equal(_np_t(p), _np_t(g))
    C = pkv.header_constants()
    for field, where, value, code in (("kept", (1, 1, 5), 40, "PKV_DEV_BAD_KEPT_INDEX"),
                                      ("sbt", (2, int(layers[1]["kept"][2, 0, 0]) >> 4), 10 ** 6,
                                       "PKV_DEV_BAD_BLOCK_ID"),  # the block of a kept token
                                      ("dbt", (0, 2), 10 ** 6, "PKV_DEV_BAD_BLOCK_ID")):
        c = dict(layers[1])
        pools, dbt = dsts[1]
        if field == "dbt":
            dbt = dbt.clone()
            dbt[where] = value
        else:
            c[field] = c[field].clone()
            c[field][where] = value
        err = pkv.new_error_word(DEV)
        torch.cuda.synchronize()
        _compact_call(c, pools, dbt, q8, True, err)
        torch.cuda.synchronize()
        assert pkv.read_error(err) == C[code], field


def test_llama8b_headline_graph_full_size():
    """The headline's launch configuration: llama8b-shaped layers (full size) over four pool
    copies, fused append + decode declaring inputs ready, captured in one CUDA graph: every
    output equal bit for bit to the eager undeclared call, pools holding the appended rows, and
    sampled rows of one layer within the gate of the oracle."""
    wl = W.WORKLOADS["llama8b"]
    cases = [W.make_layer(wl, layer=r, device=DEV, device_rng=True) for r in range(4)]
    need = pkv.decode_workspace_bytes(wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                      cases[0]["num_blocks"], cases[0]["max_blocks_per_seq"])
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    pools0 = [(c["k_cache"].clone(), c["v_cache"].clone()) for c in cases]
    eager = [_append_call(c, torch.empty_like(c["q"]), ws, False).clone() for c in cases]
    torch.cuda.synchronize()
    appended = [(c["k_cache"].clone(), c["v_cache"].clone()) for c in cases]
    for c, (k0, v0) in zip(cases, pools0):
        c["k_cache"].copy_(k0)
        c["v_cache"].copy_(v0)
    outs = [torch.full_like(c["q"], float("nan")) for c in cases]
    s = torch.cuda.Stream(DEV)
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            for c, o in zip(cases, outs):
                _append_call(c, o, ws, True, stream=s)
        graph.replay()
        torch.cuda.synchronize()
    for i, (c, o, e, (ka, va)) in enumerate(zip(cases, outs, eager, appended)):
        assert torch.equal(o, e), f"copy {i}"
        assert torch.equal(c["k_cache"], ka) and torch.equal(c["v_cache"], va)
    rows = _sample_rows(wl.batch, wl.num_q_heads, 24, seed=61)
    ref = _oracle(cases[2], rows=rows, kc=bits(appended[2][0]), vc=bits(appended[2][1]))
    assert_attn_close(outs[2].view(-1, wl.head_dim)[torch.tensor(rows, device=DEV)], ref, "llama8b graph, copy 2")


def test_sparse_layers_flagged_pipeline_full_size():
    """Two sparse layers of the layer-wise sparse workload at full size, as the bench runs them:
    the selections declaring their scores ready back to back, the first compaction undeclared
    (it follows the selections) and the second declared, and each layer's gather decode
    declared; every result equal bit for bit to the undeclared pipeline, the kept lists to the
    oracle's, and sampled rows of the second layer within the gate of the oracle."""
    wl = W.WORKLOADS["sparse"]
    lens = W.context_lengths(wl)
    layers = [W.make_layer(wl, layer=l, device=DEV, device_rng=True) for l in (4, 5)]
    scores = [W.make_scores(wl, l, lens, device=DEV, device_rng=True) for l in (4, 5)]
    dbt, dnb = W.compact_tables(wl.keep_max, wl.batch, seed=5)
    dbt = dbt.to(DEV)
    K, hkv, d = wl.keep_max, wl.num_kv_heads, wl.head_dim
    ws = torch.zeros(pkv.sparse_decode_workspace_bytes(wl.batch, wl.num_q_heads, hkv, d, layers[0]["num_blocks"],
                                                       layers[0]["max_blocks_per_seq"], K),
                     dtype=torch.uint8, device=DEV)

    def pipeline(flagged):
        err = pkv.new_error_word(DEV)
        kept = [pkv.kv_select_topk(sc, c["context_lens"], wl.n_sink, wl.n_recent, wl.k_top, error_word=err,
                                   inputs_ready=flagged) for sc, c in zip(scores, layers)]
        comp = []
        for i, (c, (kp, kl)) in enumerate(zip(layers, kept)):
            dk = torch.zeros((dnb, hkv, 16, d), dtype=torch.bfloat16, device=DEV)  # untouched slots stay 0
            dv = torch.zeros_like(dk)
            pkv.kv_compact(dk, dv, dbt, c["k_cache"], c["v_cache"], c["block_tables"], c["context_lens"], kp, kl,
                           error_word=err, inputs_ready=flagged and i > 0)
            comp.append((dk, dv))
        outs = [pkv.sparse_decode_attention(c["q"], c["k_cache"], c["v_cache"], c["block_tables"], c["context_lens"],
                                            kp, kl, wl.scale, workspace=ws, error_word=err, inputs_ready=flagged)
                .clone() for c, (kp, kl) in zip(layers, kept)]
        torch.cuda.synchronize()
        assert pkv.read_error(err) == 0
        return kept, comp, outs

    kf, cf, of = pipeline(True)
    kp_, cp_, op_ = pipeline(False)
    for i in range(2):
        okl = kp_[i][1].cpu().numpy()
        for b in range(wl.batch):
            assert torch.equal(kf[i][0][b, :, :int(okl[b])], kp_[i][0][b, :, :int(okl[b])])
        assert torch.equal(kf[i][1], kp_[i][1])
        assert torch.equal(cf[i][0], cp_[i][0]) and torch.equal(cf[i][1], cp_[i][1])
        assert torch.equal(of[i], op_[i])
    okept, okl = oracle.select_topk(scores[1].cpu().numpy(), lens.numpy(), wl.n_sink, wl.n_recent, wl.k_top)
    assert np.array_equal(kf[1][0].cpu().numpy(), okept) and np.array_equal(kf[1][1].cpu().numpy(), okl)
    rows = sorted({0, 31, 257, 511} | set(range(16 * 32 - 3, 16 * 32)))
    c = layers[1]
    ref = oracle.sparse_decode(bits(c["q"]), bits(c["k_cache"]), bits(c["v_cache"]), c["block_tables"].cpu().numpy(),
                               lens.numpy(), okept, okl, wl.scale, rows=rows)
    assert_attn_close(of[1].view(-1, d)[torch.tensor(rows, device=DEV)], ref, "sparse layer 5, flagged gather")


def _admit_layer_state(B, hkv, d, cap, seed, q8):
    """One sparse layer's rolling state: a compact pool (bf16, or INT8 codes and scales) with
    noise in unused slots, its shuffled table, and empty slot arrays."""
    rng = np.random.default_rng(seed)
    mb = (cap + 15) // 16
    nb = B * mb + 5
    st = {"bt": torch.from_numpy(rng.permutation(nb)[: B * mb].reshape(B, mb).astype(np.int32)).to(DEV),
          "slot_pos": torch.full((B, hkv, cap), -1, dtype=torch.int32, device=DEV),
          "slot_score": torch.zeros((B, hkv, cap), dtype=torch.float32, device=DEV),
          "kept_lens": torch.zeros(B, dtype=torch.int32, device=DEV)}
    if q8:
        for name in ("kq", "vq"):
            st[name] = torch.from_numpy(stored_codes(rng.integers(-127, 128, size=(nb, hkv, 16, d)))).to(DEV)
        for name in ("ks", "vs"):
            st[name] = torch.from_numpy(rng.exponential(size=(nb, hkv, 16)).astype(np.float32)).to(DEV)
    else:
        for name in ("kc", "vc"):
            st[name] = torch.from_numpy(rng.integers(0, 1 << 16, size=(nb, hkv, 16, d)).astype(np.uint16)).to(DEV) \
                .view(torch.bfloat16)
    return st


_POOL_KEYS = {False: ("kc", "vc"), True: ("kq", "vq", "ks", "vs")}
_SLOT_KEYS = ("slot_pos", "slot_score", "kept_lens")


def _admit_gpu(st, lens, kn, vn, n_sink, n_recent, q8, ready, err=None):
    if q8:
        pkv.kv_rolling_admit_q8(st["kq"], st["vq"], st["ks"], st["vs"], st["bt"], st["slot_pos"], st["slot_score"],
                                st["kept_lens"], lens, kn, vn, n_sink, n_recent, error_word=err, inputs_ready=ready)
    else:
        pkv.kv_rolling_admit(st["kc"], st["vc"], st["bt"], st["slot_pos"], st["slot_score"], st["kept_lens"], lens,
                             kn, vn, n_sink, n_recent, error_word=err, inputs_ready=ready)


def _admit_oracle(ref, bt, lens, kn, vn, n_sink, n_recent, q8):
    """The oracle's admission on numpy state `ref` (pool arrays then the slot arrays), in place."""
    if q8:
        out = oracle.rolling_admit_q8(*(ref[k] for k in ("kq", "vq", "ks", "vs")), bt, ref["slot_pos"],
                                      ref["slot_score"], ref["kept_lens"], lens, kn, vn, n_sink, n_recent)
        keys = ("kq", "vq", "ks", "vs") + _SLOT_KEYS
    else:
        out = oracle.rolling_admit(ref["kc"], ref["vc"], bt, ref["slot_pos"], ref["slot_score"], ref["kept_lens"],
                                   lens, kn, vn, n_sink, n_recent)
        keys = ("kc", "vc") + _SLOT_KEYS
    ref.update(zip(keys, out))


@pytest.mark.parametrize("q8,d", [(False, 128), (False, 64), (True, 128)])
def test_admissions_of_interleaved_layers_flagged_against_oracle(q8, d):
    """PKV_ADMIT_INPUTS_READY: three sparse layers, each with its own rolling state, stepped from
    empty to full and past it with no synchronisation: per step, each layer's admission (flagged)
    and then that layer's score update (a torch add standing in for its score pass), so each
    admission's preceding work is the previous layer's update, never its own state's writer.  The
    final state of every layer equals the oracle's chain bit for bit."""
    B, hkv, n_sink, k_top, n_recent = 3, 4, 4, 24, 32
    cap = n_sink + k_top + n_recent
    layers = [_admit_layer_state(B, hkv, d, cap, 90 + 7 * l, q8) for l in range(3)]
    rng = np.random.default_rng(5 + d)
    g = torch.Generator().manual_seed(6 + d)
    steps = 110
    kns = [[rand_bf16((B, hkv, d), g) for _ in layers] for _ in range(steps)]
    vns = [[rand_bf16((B, hkv, d), g) for _ in layers] for _ in range(steps)]
    incs = [[rng.choice([0.0, 0.25, 0.5, 1.0], size=(B, hkv, cap)).astype(np.float32) for _ in layers]
            for _ in range(steps)]
    lens = [torch.full((B,), L, dtype=torch.int32, device=DEV) for L in range(1, steps + 1)]
    refs = [{k: v.cpu().numpy().copy() if v.dtype != torch.bfloat16 else bits(v) for k, v in st.items() if k != "bt"}
            for st in layers]
    dk = [[(kns[i][l].to(DEV), vns[i][l].to(DEV), torch.from_numpy(incs[i][l]).to(DEV)) for l in range(3)]
          for i in range(steps)]
    err = pkv.new_error_word(DEV)
    torch.cuda.synchronize()
    for i in range(steps):
        for l, st in enumerate(layers):
            kn, vn, inc = dk[i][l]
            _admit_gpu(st, lens[i], kn, vn, n_sink, n_recent, q8, True, err)
            st["slot_score"].add_(inc)
    torch.cuda.synchronize()
    assert pkv.read_error(err) == 0
    for l, (st, ref) in enumerate(zip(layers, refs)):
        bt = st["bt"].cpu().numpy()
        for i in range(steps):
            _admit_oracle(ref, bt, lens[i].cpu().numpy(), bits(kns[i][l]), bits(vns[i][l]), n_sink, n_recent, q8)
            ref["slot_score"] = ref["slot_score"] + incs[i][l]
        for name in _POOL_KEYS[q8] + _SLOT_KEYS:
            got = st[name]
            got = bits(got) if got.dtype == torch.bfloat16 else got.cpu().numpy()
            assert np.array_equal(got, ref[name]), f"layer {l} {name}"


def test_admission_flagged_errors_after_the_wait():
    """A NaN slot score and a context length of 0, found before the wait by flagged admissions,
    are recorded once the calls may write; the (b, g) with the NaN and the sequence with the bad
    length are left unchanged."""
    B, hkv, d, n_sink, k_top, n_recent = 2, 2, 64, 2, 4, 6
    cap = n_sink + k_top + n_recent
    st = _admit_layer_state(B, hkv, d, cap, 31, False)
    g = torch.Generator().manual_seed(31)
    for L in range(1, cap + 1):  # fill the budget
        _admit_gpu(st, torch.full((B,), L, dtype=torch.int32, device=DEV), rand_bf16((B, hkv, d), g).to(DEV),
                   rand_bf16((B, hkv, d), g).to(DEV), n_sink, n_recent, False, False)
    torch.cuda.synchronize()
    st["slot_score"][1, 0, 5] = float("nan")
    before = {k: st[k].clone() for k in ("slot_pos", "slot_score", "kept_lens")}
    err = pkv.new_error_word(DEV)
    torch.cuda.synchronize()
    _admit_gpu(st, torch.full((B,), cap + 1, dtype=torch.int32, device=DEV), rand_bf16((B, hkv, d), g).to(DEV),
               rand_bf16((B, hkv, d), g).to(DEV), n_sink, n_recent, False, True, err)
    torch.cuda.synchronize()
    C = pkv.header_constants()
    assert pkv.read_error(err, clear=True) == C["PKV_DEV_BAD_SCORE"]
    assert torch.equal(st["slot_pos"][1, 0], before["slot_pos"][1, 0])
    assert not torch.equal(st["slot_pos"][0, 0], before["slot_pos"][0, 0])   # the others admitted
    st["slot_score"][1, 0, 5] = 0.0
    before = {k: st[k].clone() for k in ("slot_pos", "slot_score", "kept_lens")}
    torch.cuda.synchronize()
    bad = torch.tensor([cap + 2, 0], dtype=torch.int32, device=DEV)
    _admit_gpu(st, bad, rand_bf16((B, hkv, d), g).to(DEV), rand_bf16((B, hkv, d), g).to(DEV), n_sink, n_recent,
               False, True, err)
    torch.cuda.synchronize()
    assert pkv.read_error(err) == C["PKV_DEV_BAD_CONTEXT_LEN"]
    assert torch.equal(st["slot_pos"][1], before["slot_pos"][1]) and torch.equal(st["kept_lens"], before["kept_lens"])
