"""GPU parity of the prefill-window score (pkv_prefill_window_scores) against the fp64 oracle
(oracle.prefill_scores).  d = 128 with G a power of two runs the tcgen05 kernel, d = 64 and
G = 6 the warp-level one; both are covered.

Tolerances: each probability is exp2 of an fp32 logit (exact bf16 products, fp32 sums) minus an
fp32 log-sum-exp, so it carries a relative error of ~1e-6 (the logit's fp32 error times its
magnitude); a key's score sums at most alpha * G of them in fp32.  Scores must match to 2e-4
relative + 1e-7 absolute, the computed lse to 1e-4 absolute + 1e-5 relative.  A segment's
scores sum to G times its window rows, which checks every segment at full size."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_mapped_gb300 as pkv
from paged_kv_cache_mapped_gb300 import inputs as W
from helpers import bits, paged_from_contiguous, rand_bf16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
RTOL, ATOL = 2e-4, 1e-7


def _case(lens, alpha, hq, hkv, d, seed, nb_extra=5):
    g = torch.Generator().manual_seed(seed)
    B = len(lens)
    lmax = max(max(lens), 1)
    k = rand_bf16((B, lmax, hkv, d), g)
    v = rand_bf16((B, lmax, hkv, d), g)
    q = rand_bf16((B, alpha, hq, d), g)
    nb = sum((L + 15) // 16 for L in lens) + nb_extra
    kc, _, bt = paged_from_contiguous(k, v, lens, nb, g)
    return {"q": q.to(DEV), "kc": kc.to(DEV), "bt": bt.to(DEV),
            "lens": torch.tensor(lens, dtype=torch.int32, device=DEV), "alpha": alpha, "scale": d ** -0.5}


def _gpu(c, stride, init=None, lse=None, lse_given=False, err=None):
    B, _, hq, _ = c["q"].shape
    hkv = c["kc"].shape[1]
    acc = torch.zeros((B, hkv, stride), dtype=torch.float32, device=DEV) if init is None else init.clone()
    before = acc.clone()
    lse = pkv.prefill_window_scores(c["q"], c["kc"], c["bt"], c["lens"], c["scale"], acc, lse=lse,
                                    lse_given=lse_given, error_word=err)
    torch.cuda.synchronize()
    return (acc - before).double().cpu().numpy(), lse


def _ref(c, stride, lse=None, segs=None):
    return oracle.prefill_scores(bits(c["q"]), bits(c["kc"]), c["bt"].cpu().numpy(), c["lens"].cpu().numpy(),
                                 c["alpha"], c["scale"], lse=lse, stride=stride, segs=segs)


def _check(got, ref, what):
    bad = np.abs(got - ref) > RTOL * np.abs(ref) + ATOL
    assert not bad.any(), f"{what}: {bad.sum()} scores off, worst {np.abs(got - ref).max():.3e}"


def _check_lse(got, ref, what):
    g = got.double().cpu().numpy()
    ok = np.isclose(g, ref, rtol=1e-5, atol=1e-4) | (np.isneginf(g) & np.isneginf(ref))
    assert ok.all(), f"{what}: lse off"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("group", [1, 4, 6, 8])
def test_ragged_prompts_all_groups(d, group):
    hkv = 2
    lens = [300, 17, 0, 1, 129, 64, 200]
    alpha = 40
    c = _case(lens, alpha, hkv * group, hkv, d, seed=d + group)
    stride = 304
    got, lse = _gpu(c, stride)
    ref, ref_lse = _ref(c, stride)
    _check(got, ref, f"d={d} G={group}")
    _check_lse(lse, ref_lse, f"d={d} G={group}")


@pytest.mark.parametrize("alpha", [1, 16, 64, 256])
def test_window_sizes(alpha):
    c = _case([700, 300, 90], alpha, 16, 4, 128, seed=alpha)
    stride = 704
    got, lse = _gpu(c, stride)
    ref, ref_lse = _ref(c, stride)
    _check(got, ref, f"alpha={alpha}")
    _check_lse(lse, ref_lse, f"alpha={alpha}")
    rows = np.array([min(L, alpha) for L in (700, 300, 90)], dtype=np.float64)
    np.testing.assert_allclose(got.sum(axis=2), np.repeat((4.0 * rows)[:, None], 4, axis=1), rtol=1e-4)


def test_given_lse_and_accumulation():
    c = _case([500, 130], 48, 8, 2, 128, seed=3)
    stride = 512
    _, ref_lse = _ref(c, stride)
    lse = torch.from_numpy(ref_lse.astype(np.float32)).to(DEV)
    init = torch.rand((2, 2, stride), generator=torch.Generator().manual_seed(4)).to(DEV)
    got, lse_out = _gpu(c, stride, init=init, lse=lse, lse_given=True)
    ref, _ = _ref(c, stride, lse=lse.double().cpu().numpy())
    _check(got, ref, "given lse")
    assert torch.equal(lse_out, lse)          # read, not written


@pytest.mark.parametrize("d", [64, 128])  # the warp-level kernel and the tcgen05 one
def test_bad_block_is_reported_and_skipped(d):
    c = _case([200, 90], 16, 8, 2, d, seed=5)
    c["bt"][0, 3] = 10 ** 6
    err = pkv.new_error_word(DEV)
    got, _ = _gpu(c, 208, err=err)
    assert pkv.read_error(err) == pkv.header_constants()["PKV_DEV_BAD_BLOCK_ID"]
    # the second sequence does not touch the bad entry
    ref, _ = _ref({**c, "bt": c["bt"][1:], "lens": c["lens"][1:], "q": c["q"][1:]}, 208)
    _check(got[1:], ref, "untouched sequence")


def test_sparse_layer_full_size():
    """16 prompts of 16384 tokens, 32/8 heads, d = 128, a 256-token window: every segment's sum
    against G x 256, and three segments against the oracle."""
    wl = W.WORKLOADS["sparse"]
    c0 = W.make_layer(wl, device=DEV, device_rng=True)
    B, hq, hkv, d = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    alpha = 256
    g = torch.Generator(device=DEV).manual_seed(7)
    c = {"q": torch.randn((B, alpha, hq, d), generator=g, device=DEV).to(torch.bfloat16), "kc": c0["k_cache"],
         "bt": c0["block_tables"], "lens": c0["context_lens"], "alpha": alpha, "scale": wl.scale}
    stride = c0["max_blocks_per_seq"] * 16
    err = pkv.new_error_word(DEV)
    got, lse = _gpu(c, stride, err=err)
    assert pkv.read_error(err) == 0
    np.testing.assert_allclose(got.sum(axis=2), np.full((B, hkv), 4.0 * alpha), rtol=2e-4)
    segs = [0, 37, B * hkv - 1]
    ref, ref_lse = _ref(c, stride, segs=segs)
    _check(got.reshape(-1, stride)[segs], ref, "sparse layer")
    heads = [h for s in segs for h in range((s % hkv) * 4, (s % hkv) * 4 + 4)]
    bs = [s // hkv for s in segs for _ in range(4)]
    _check_lse(lse[bs, heads], ref_lse[bs, heads], "sparse layer lse")
