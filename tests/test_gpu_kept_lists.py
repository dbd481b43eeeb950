"""Kept lists on the GPU: the gather form of the sparse decode and the compaction over lists of
the shapes a sparse layer produces, and both hold every list to its contract (entries strictly
ascending inside [0, L_b): each retained token is attended and copied once, "How KV Sparsity
Achieves 1.5x Acceleration for vLLM", section "System model").

- Lists built from sink, scattered and recent-window positions, contiguous runs at every offset,
  lengths of every residue mod 16 and the short and empty cases, for bf16 and INT8 pools at
  d = 64 and 128: every output element against the fp64 oracle (attention gate).
- Lists with a duplicated or a descending entry: the call reports PKV_DEV_BAD_KEPT_INDEX, and the
  rows of every other (sequence, kv head) equal the oracle's on the uncorrupted lists (attention
  gate for the decode, bit for bit for the compaction)."""
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


def _pools(lens, hq, hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    B, lmax = len(lens), max(max(lens), 1)
    k, v = rand_bf16((B, lmax, hkv, d), g), rand_bf16((B, lmax, hkv, d), g)
    nb = sum((L + 15) // 16 for L in lens) + 4
    kc, vc, bt = paged_from_contiguous(k, v, lens, nb, g, fill=float("nan"))
    return {"q": rand_bf16((B, hq, d), g), "kc": kc, "vc": vc, "bt": bt,
            "lens": torch.tensor(lens, dtype=torch.int32), "scale": d ** -0.5}


def _structured_list(L, kind, rng):
    """Ascending positions in [0, L) of one shape of kept list."""
    if kind == "sink_topk_recent":      # the sparse layer's shape: 4 sinks, scattered, a window
        recent = min(L, int(rng.integers(16, 200)))
        mid = np.arange(4, max(4, L - recent))
        top = rng.choice(mid, size=min(len(mid), int(rng.integers(0, 60))), replace=False) if len(mid) else []
        pos = set(range(min(4, L))) | set(int(x) for x in top) | set(range(L - recent, L))
    elif kind == "runs":                # contiguous runs starting at every residue
        pos = set()
        start = int(rng.integers(0, 16))
        while start < L:
            run = int(rng.integers(1, 70))
            pos |= set(range(start, min(L, start + run)))
            start += run + int(rng.integers(1, 40))
    elif kind == "all":                 # every token: all whole blocks but the tail
        pos = set(range(L))
    elif kind == "scattered":
        pos = set(int(x) for x in rng.choice(L, size=min(L, int(rng.integers(1, 100))), replace=False))
    else:                               # "window": only the last tokens (a sliding window)
        pos = set(range(max(0, L - int(rng.integers(1, 300))), L))
    return np.array(sorted(pos), dtype=np.int32)


def _lists(lens, hkv, kinds, seed):
    """kept [B, Hkv, max_kept], kept_lens [B]: every kv head of a sequence keeps the same count,
    so each head's list is one shape cut (or padded with unique positions) to that count."""
    rng = np.random.default_rng(seed)
    per = []
    for b, L in enumerate(lens):
        heads = [_structured_list(L, kinds[(b + gh) % len(kinds)], rng) if L > 0 else np.zeros(0, np.int32)
                 for gh in range(hkv)]
        per.append(heads)
    counts = [min(len(h) for h in heads) for heads in per]
    max_kept = max(max(counts), 1)
    kept = np.full((len(lens), hkv, max_kept), -1, dtype=np.int32)
    for b, heads in enumerate(per):
        for gh, h in enumerate(heads):
            kept[b, gh, :counts[b]] = h[len(h) - counts[b]:]   # keep the list's tail (the window side)
    return kept, np.array(counts, dtype=np.int32)


LENS = [1, 15, 16, 17, 33, 100, 255, 256, 257, 1000, 1031, 2047, 0, 4093]


def _gather(c, kept, kl, q8, err):
    dv = lambda t: t.to(DEV)
    if q8:
        return pkv.sparse_decode_attention_q8(dv(c["q"]), dv(c["kq"]), dv(c["vq"]), dv(c["ks"]), dv(c["vs"]),
                                              dv(c["bt"]), dv(c["lens"]), dv(torch.from_numpy(kept)),
                                              dv(torch.from_numpy(kl)), c["scale"], error_word=err)
    return pkv.sparse_decode_attention(dv(c["q"]), dv(c["kc"]), dv(c["vc"]), dv(c["bt"]), dv(c["lens"]),
                                       dv(torch.from_numpy(kept)), dv(torch.from_numpy(kl)), c["scale"],
                                       error_word=err)


def _oracle(c, kept, kl, q8, rows=None):
    if q8:
        return oracle.sparse_decode_q8(bits(c["q"]), c["kq"].numpy(), c["ks"].numpy(), c["vq"].numpy(),
                                       c["vs"].numpy(), c["bt"].numpy(), c["lens"].numpy(), kept, kl, c["scale"],
                                       rows=rows)
    return oracle.sparse_decode(bits(c["q"]), bits(c["kc"]), bits(c["vc"]), c["bt"].numpy(), c["lens"].numpy(),
                                kept, kl, c["scale"], rows=rows)


def _with_q8(c):
    # INT8 pools from the bf16 ones (the NaN rows outside the contexts become zero rows)
    kc = torch.nan_to_num(c["kc"].float()).to(torch.bfloat16)
    vc = torch.nan_to_num(c["vc"].float()).to(torch.bfloat16)
    kq, ks = oracle.quantize_rows(bits(kc))
    vq, vs = oracle.quantize_rows(bits(vc))
    c.update(kq=torch.from_numpy(kq), ks=torch.from_numpy(ks), vq=torch.from_numpy(vq), vs=torch.from_numpy(vs))
    return c


def _close(got, ref, q8, what):
    if q8:  # the INT8 decode's gate: outputs relative to max(1, max |ref|)
        top = max(1.0, float(np.abs(ref).max()) if ref.size else 1.0)
        assert_attn_close(got.float() / top, ref / top, what)
    else:
        assert_attn_close(got, ref, what)


@pytest.mark.parametrize("q8", [False, True])
@pytest.mark.parametrize("d,hq,hkv", [(128, 16, 4), (64, 6, 2)])
@pytest.mark.parametrize("kinds", [("sink_topk_recent",), ("runs", "all", "window"), ("scattered", "runs")])
def test_gather_whole_blocks_and_rows_against_oracle(q8, d, hq, hkv, kinds):
    c = _pools(LENS, hq, hkv, d, seed=d + hq + len(kinds[0]))
    if q8:
        c = _with_q8(c)
    kept, kl = _lists(LENS, hkv, kinds, seed=7 * d + len(kinds))
    err = pkv.new_error_word(DEV)
    out = _gather(c, kept, kl, q8, err)
    torch.cuda.synchronize()
    assert pkv.read_error(err) == 0
    _close(out, _oracle(c, kept, kl, q8), q8, f"{'int8' if q8 else 'bf16'} d={d} {kinds}")


def test_gather_full_size_sparse_layer():
    """The sparse workload's layer at full size (1540 kept of 16384: 4 sinks, 512 top-scored, the
    1024 most recent) against the oracle on sampled rows, and the same lists cut one entry short
    (a partial last unit in every list)."""
    wl = W.WORKLOADS["sparse"]
    lens = W.context_lengths(wl)
    case = W.make_layer(wl, layer=5, device=DEV, device_rng=True)
    scores = W.make_scores(wl, 5, lens, device=DEV, device_rng=True)
    okept, okl = oracle.select_topk(scores.cpu().numpy(), lens.numpy(), wl.n_sink, wl.n_recent, wl.k_top)
    rows = sorted({0, 7, 31, 64, 255, 300, 511} | set(range(16 * 32 - 3, 16 * 32)))
    idx = torch.tensor(rows, device=DEV)
    for cut in (0, 1):
        kl = (okl - cut).astype(np.int32)
        err = pkv.new_error_word(DEV)
        out = pkv.sparse_decode_attention(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                                          case["context_lens"], torch.from_numpy(okept).to(DEV),
                                          torch.from_numpy(kl).to(DEV), wl.scale, error_word=err)
        torch.cuda.synchronize()
        assert pkv.read_error(err) == 0
        ref = oracle.sparse_decode(bits(case["q"]), bits(case["k_cache"]), bits(case["v_cache"]),
                                   case["block_tables"].cpu().numpy(), lens.numpy(), okept, kl, wl.scale, rows=rows)
        assert_attn_close(out.view(-1, 128)[idx], ref, f"sparse layer, lists cut by {cut}")


def _corrupt(kept, kl):
    """Duplicate one entry of (1, 0) and put a descent into (2, 1); returns the corrupted copy
    and the (b, g) pairs touched."""
    bad = kept.copy()
    assert kl[1] >= 2 and kl[2] >= 2
    i, m = min(5, int(kl[1]) - 1), int(kl[2]) // 2
    bad[1, 0, i] = bad[1, 0, i - 1]                          # a duplicate
    bad[2, 1, m - 1], bad[2, 1, m] = bad[2, 1, m], bad[2, 1, m - 1]  # a descent
    return bad, {(1, 0), (2, 1)}


def _valid_rows(B, hq, hkv, touched):
    G = hq // hkv
    return [b * hq + h for b in range(B) for h in range(hq) if (b, h // G) not in touched]


@pytest.mark.parametrize("q8", [False, True])
def test_gather_rejects_duplicates_and_descents(q8):
    lens = [300, 700, 1200, 90]
    hq, hkv, d = 8, 2, 128
    c = _pools(lens, hq, hkv, d, seed=61)
    if q8:
        c = _with_q8(c)
    kept, kl = _lists(lens, hkv, ("sink_topk_recent", "runs"), seed=62)
    bad, touched = _corrupt(kept, kl)
    err = pkv.new_error_word(DEV)
    out = _gather(c, bad, kl, q8, err)
    torch.cuda.synchronize()
    assert pkv.read_error(err) == C["PKV_DEV_BAD_KEPT_INDEX"]
    assert torch.isfinite(out.float()).all()
    rows = _valid_rows(len(lens), hq, hkv, touched)
    ref = _oracle(c, kept, kl, q8, rows=rows)
    _close(out.view(-1, d)[torch.tensor(rows, device=DEV)], ref, q8, "untouched segments")


@pytest.mark.parametrize("q8", [False, True])
def test_compaction_rejects_duplicates_and_descents(q8):
    lens = [300, 700, 1200, 90]
    hq, hkv, d = 8, 2, 128
    c = _pools(lens, hq, hkv, d, seed=63)
    if q8:
        c = _with_q8(c)
    kept, kl = _lists(lens, hkv, ("sink_topk_recent", "runs"), seed=64)
    bad, touched = _corrupt(kept, kl)
    B = len(lens)
    dbt, dnb = W.compact_tables(kept.shape[2], B, seed=65)
    err = pkv.new_error_word(DEV)
    dv = lambda t: t.to(DEV)
    if q8:
        z = lambda: torch.zeros((dnb, hkv, 16, d), dtype=torch.uint8)
        zs = lambda: torch.zeros((dnb, hkv, 16), dtype=torch.float32)
        dst = [z(), z(), zs(), zs()]
        ref = oracle.compact_q8(dst[0].numpy(), dst[1].numpy(), dst[2].numpy(), dst[3].numpy(), dbt.numpy(),
                                c["kq"].numpy(), c["vq"].numpy(), c["ks"].numpy(), c["vs"].numpy(), c["bt"].numpy(),
                                c["lens"].numpy(), kept, kl)
        got = [dv(t) for t in dst]
        pkv.kv_compact_q8(*got, dv(dbt), dv(c["kq"]), dv(c["vq"]), dv(c["ks"]), dv(c["vs"]), dv(c["bt"]),
                          dv(c["lens"]), dv(torch.from_numpy(bad)), dv(torch.from_numpy(kl)), error_word=err)
        got = [t.cpu().numpy() for t in got]
    else:
        dk = torch.zeros((dnb, hkv, 16, d), dtype=torch.bfloat16)
        dvv = torch.zeros_like(dk)
        ref = oracle.compact(bits(dk), bits(dvv), dbt.numpy(), bits(c["kc"]), bits(c["vc"]), c["bt"].numpy(),
                             c["lens"].numpy(), kept, kl)
        gk, gv = dv(dk), dv(dvv)
        pkv.kv_compact(gk, gv, dv(dbt), dv(c["kc"]), dv(c["vc"]), dv(c["bt"]), dv(c["lens"]),
                       dv(torch.from_numpy(bad)), dv(torch.from_numpy(kl)), error_word=err)
        got = [bits(gk), bits(gv)]
    assert pkv.read_error(err) == C["PKV_DEV_BAD_KEPT_INDEX"]
    # every untouched (b, g): its compact rows equal the oracle's bit for bit
    dbt_n = dbt.numpy()
    for b in range(B):
        for g in range(hkv):
            if (b, g) in touched:
                continue
            for j in range(int(kl[b])):
                blk, off = dbt_n[b, j // 16], j % 16
                for gt, rf in zip(got, ref):
                    assert np.array_equal(gt[blk, g, off], rf[blk, g, off]), (b, g, j)
