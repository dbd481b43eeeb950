"""GPU parity of the score-emitting decode (pkv_paged_decode_attention_scores) against the fp64
oracle (oracle.decode_scores).

Tolerances: the GPU logits are fp32 dot products of exact bf16 products (relative error
~1e-6), turned into probabilities with exp2 and a log-sum-exp kept in fp32, so every score
increment matches the fp64 value to a relative 5e-4 (bound taken with a wide margin; the
attention output keeps its own max-abs 1e-2 / rel-L2 2e-3 gate and is in fact bit-identical to
the plain decode's).  Row log-sum-exps match to 1e-4 absolute + 1e-5 relative.  Each row's
probabilities sum to 1, so a (sequence, kv head)'s increments sum to G."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_mapped_gb300 as pkv
from paged_kv_cache_mapped_gb300 import inputs as W
from helpers import bits, paged_from_contiguous, rand_bf16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
RTOL, ATOL = 5e-4, 1e-7


def _small_case(lens, hq, hkv, d, seed, nb_extra=5):
    g = torch.Generator().manual_seed(seed)
    B = len(lens)
    lmax = max(max(lens), 1)
    k = rand_bf16((B, lmax, hkv, d), g)
    v = rand_bf16((B, lmax, hkv, d), g)
    q = rand_bf16((B, hq, d), g)
    nb = sum((L + 15) // 16 for L in lens) + nb_extra
    kc, vc, bt = paged_from_contiguous(k, v, lens, nb, g)
    return {"q": q.to(DEV), "k_cache": kc.to(DEV), "v_cache": vc.to(DEV), "block_tables": bt.to(DEV),
            "context_lens": torch.tensor(lens, dtype=torch.int32, device=DEV), "scale": d ** -0.5}


def _run_scores(case, stride, window=0, init=None, err=None, **kw):
    B, hq, d = case["q"].shape
    hkv = case["k_cache"].shape[1]
    acc = (torch.zeros if init is None else (lambda *a, **k: init.clone()))((B, hkv, stride), dtype=torch.float32,
                                                                            device=DEV)
    before = acc.clone()
    out, lse = pkv.paged_decode_attention_scores(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                                                 case["context_lens"], case["scale"], acc, window,
                                                 error_word=err, **kw)
    torch.cuda.synchronize()
    return out, lse, (acc - before).double().cpu().numpy(), acc


def _oracle(case, stride, window=0, segs=None):
    return oracle.decode_scores(bits(case["q"]), bits(case["k_cache"]), case["block_tables"].cpu().numpy(),
                                case["context_lens"].cpu().numpy(), case["scale"], window, stride=stride,
                                segs=segs)


def _check_scores(got, ref, what):
    bad = np.abs(got - ref) > RTOL * np.abs(ref) + ATOL
    assert not bad.any(), f"{what}: {bad.sum()} scores off, worst {np.abs(got - ref).max():.3e}"


def _check_lse(got, ref, what):
    ok = np.isclose(got, ref, rtol=1e-5, atol=1e-4) | (np.isneginf(got) & np.isneginf(ref))
    assert ok.all(), f"{what}: lse off by {np.nanmax(np.abs(np.where(np.isfinite(ref), got - ref, 0)))}"


@pytest.mark.parametrize("window", [0, 1, 16, 50, 300])
def test_tiny_workload_every_score(window):
    case = W.make_layer(W.WORKLOADS["tiny"], device=DEV)
    stride = 260
    g = torch.Generator().manual_seed(7)
    init = torch.rand((2, 8, stride), generator=g).to(DEV)
    err = pkv.new_error_word(DEV)
    out, lse, delta, acc = _run_scores(case, stride, window, init=init, err=err)
    assert pkv.read_error(err) == 0
    ref, ref_lse = _oracle(case, stride, window)
    _check_scores(delta, ref, f"tiny window={window}")
    _check_lse(lse.double().cpu().numpy(), ref_lse, f"tiny window={window}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("group", [1, 4, 6, 8])
def test_ragged_lengths_all_groups(d, group):
    hkv = 2
    lens = [700, 1, 0, 33, 1500, 16, 257]
    case = _small_case(lens, hkv * group, hkv, d, seed=d + group)
    stride = 1504
    out, lse, delta, _ = _run_scores(case, stride)
    ref, ref_lse = _oracle(case, stride)
    _check_scores(delta, ref, f"d={d} G={group}")
    _check_lse(lse.double().cpu().numpy(), ref_lse, f"d={d} G={group}")
    sums = delta.sum(axis=2)
    expect = np.array([[group if L > 0 else 0] * hkv for L in lens], dtype=np.float64)
    np.testing.assert_allclose(sums, expect, rtol=1e-4, atol=1e-6)


def test_output_bit_identical_to_plain_decode_and_append():
    case = _small_case([900, 33, 1500, 129], hq=16, hkv=4, d=128, seed=11)
    plain = pkv.paged_decode_attention(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                                       case["context_lens"], case["scale"]).clone()
    out, _, _, _ = _run_scores(case, 1504)
    assert torch.equal(out, plain)
    # with this step's append: same pool update and output as the fused append entry point
    g = torch.Generator().manual_seed(12)
    k_new = rand_bf16((4, 4, 128), g).to(DEV)
    v_new = rand_bf16((4, 4, 128), g).to(DEV)
    kc0, vc0 = case["k_cache"].clone(), case["v_cache"].clone()
    ref_out = pkv.paged_decode_attention_append(case["q"], case["k_cache"], case["v_cache"], k_new, v_new,
                                                case["block_tables"], case["context_lens"], case["scale"]).clone()
    kc1, vc1 = case["k_cache"].clone(), case["v_cache"].clone()
    case["k_cache"].copy_(kc0)
    case["v_cache"].copy_(vc0)
    out, _, delta, _ = _run_scores(case, 1504, k_new=k_new, v_new=v_new)
    assert torch.equal(out, ref_out)
    assert torch.equal(case["k_cache"], kc1) and torch.equal(case["v_cache"], vc1)
    ref, _ = _oracle(case, 1504)  # the pools now hold the appended rows
    _check_scores(delta, ref, "append")


def _sample_segs(B, hkv, n, seed):
    rng = np.random.default_rng(seed)
    segs = {0, B * hkv - 1} | set(rng.choice(B * hkv, size=min(n, B * hkv), replace=False).tolist())
    return sorted(segs)


def test_llama8b_full_size_sampled_segments():
    wl = W.WORKLOADS["llama8b"]
    case = W.make_layer(wl, device=DEV, device_rng=True)
    stride = case["max_blocks_per_seq"] * 16
    err = pkv.new_error_word(DEV)
    out, lse, delta, _ = _run_scores(case, stride, err=err)
    assert pkv.read_error(err) == 0
    np.testing.assert_allclose(delta.sum(axis=2), np.full((wl.batch, wl.num_kv_heads), wl.group), rtol=1e-4)
    segs = _sample_segs(wl.batch, wl.num_kv_heads, 24, 31)
    ref, ref_lse = _oracle(case, stride, segs=segs)
    got = delta.reshape(-1, stride)[segs]
    _check_scores(got, ref, "llama8b")
    G = wl.group
    lse_np = lse.double().cpu().numpy().reshape(-1)
    got_lse = np.stack([lse_np[(s // wl.num_kv_heads) * wl.num_q_heads + (s % wl.num_kv_heads) * G + np.arange(G)]
                        for s in segs])
    _check_lse(got_lse, ref_lse, "llama8b")


def test_long128k_sampled_segments():
    wl = W.WORKLOADS["long128k"]
    case = W.make_layer(wl, device=DEV, device_rng=True)
    stride = 131072
    out, lse, delta, _ = _run_scores(case, stride)
    np.testing.assert_allclose(delta.sum(axis=2), np.full((wl.batch, wl.num_kv_heads), wl.group), rtol=1e-4)
    segs = [0, 13, 31]
    ref, _ = _oracle(case, stride, segs=segs)
    _check_scores(delta.reshape(-1, stride)[segs], ref, "long128k")


def test_short_score_rows_are_reported_and_bounded():
    """A context longer than the score rows: the keys beyond them get no score and the call
    reports the length.  Rows are adjacent in memory, so a write past a row would land in the
    next (sequence, kv head)'s scores and fail the comparison."""
    case = _small_case([300, 40], hq=8, hkv=2, d=64, seed=13)
    stride = 128
    err = pkv.new_error_word(DEV)
    acc = torch.zeros((2, 2, stride), dtype=torch.float32, device=DEV)
    out, lse = pkv.paged_decode_attention_scores(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                                                 case["context_lens"], case["scale"], acc, error_word=err)
    torch.cuda.synchronize()
    assert pkv.read_error(err) == pkv.header_constants()["PKV_DEV_BAD_CONTEXT_LEN"]
    ref, _ = _oracle(case, 300)
    _check_scores(acc.double().cpu().numpy(), ref[:, :, :stride], "short rows")
    plain = pkv.paged_decode_attention(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                                       case["context_lens"], case["scale"])
    assert torch.equal(out, plain)


def test_emitted_scores_feed_the_selection():
    """Scores accumulated over three decode steps (three query sets) select the kept set: the
    GPU selection on those scores equals the oracle's selection on the same scores, bit for bit."""
    lens = [3000, 1700, 2600]
    case = _small_case(lens, hq=8, hkv=2, d=128, seed=14)
    stride = 3008
    acc = torch.zeros((3, 2, stride), dtype=torch.float32, device=DEV)
    g = torch.Generator().manual_seed(15)
    for _ in range(3):
        case["q"] = rand_bf16((3, 8, 128), g).to(DEV)
        pkv.paged_decode_attention_scores(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                                          case["context_lens"], case["scale"], acc)
    n_sink, n_recent, k_top = 4, 256, 300
    kept = torch.full((3, 2, n_sink + k_top + n_recent), -7, dtype=torch.int32, device=DEV)
    kept_lens = torch.empty(3, dtype=torch.int32, device=DEV)
    err = pkv.new_error_word(DEV)
    pkv.kv_select_topk(acc, case["context_lens"], n_sink, n_recent, k_top, kept_out=kept, kept_lens_out=kept_lens,
                       error_word=err)
    assert pkv.read_error(err) == 0
    ref_kept, ref_lens = oracle.select_topk(acc.cpu().numpy(), case["context_lens"].cpu().numpy(),
                                            n_sink, n_recent, k_top)
    assert np.array_equal(kept_lens.cpu().numpy(), ref_lens)
    for b in range(3):
        n = int(ref_lens[b])
        assert np.array_equal(kept[b, :, :n].cpu().numpy(), ref_kept[b, :, :n])


def test_unaligned_score_rows_take_the_scalar_path():
    """score_stride not a multiple of 4 and buffers only 4-byte aligned: same scores."""
    case = _small_case([301, 77, 5], hq=8, hkv=2, d=64, seed=16)
    stride = 303
    big = torch.zeros((3 * 2 * stride + 1,), dtype=torch.float32, device=DEV)
    acc = big[1:].view(3, 2, stride)                       # offset by 4 bytes
    lg_big = torch.empty((3 * 8 * stride + 1,), dtype=torch.float32, device=DEV)
    logits = lg_big[1:].view(3, 8, stride)
    pkv.paged_decode_attention_scores(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                                      case["context_lens"], case["scale"], acc, 40, logits=logits)
    torch.cuda.synchronize()
    ref, _ = _oracle(case, stride, window=40)
    _check_scores(acc.double().cpu().numpy(), ref, "unaligned")
