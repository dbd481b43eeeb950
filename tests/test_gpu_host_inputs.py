"""Decode calls whose q, new K/V rows, block tables, lengths and out live in pinned host memory
(pkv_device_alias): the kernels read and write them in place over the host link, and every
result is bit-identical to the same call on device copies of those tensors -- which the other
test files check against the fp64 oracle -- and within the gate of the oracle itself here.
Covered: the fused append + decode (bf16 and INT8 pools; the pools end identical), the plain
decode with a window, the gather form of the sparse decode, the no-workspace entry point, calls
declaring their inputs ready back to back and captured in a CUDA graph, and the refusal of
pageable host memory."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_mapped_gb300 as pkv
from helpers import assert_attn_close, bits, paged_from_contiguous, rand_bf16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _case(lens, hq, hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    B, lmax = len(lens), max(max(lens), 1)
    k, v = rand_bf16((B, lmax, hkv, d), g), rand_bf16((B, lmax, hkv, d), g)
    nb = sum((L + 15) // 16 for L in lens) + 3
    kc, vc, bt = paged_from_contiguous(k, v, lens, nb, g)
    return {"q": rand_bf16((B, hq, d), g), "k_cache": kc.to(DEV), "v_cache": vc.to(DEV), "block_tables": bt,
            "context_lens": torch.tensor(lens, dtype=torch.int32), "scale": d ** -0.5,
            "k_new": rand_bf16((B, hkv, d), g), "v_new": rand_bf16((B, hkv, d), g)}


_HOST = ("q", "k_new", "v_new", "block_tables", "context_lens")


def _placed(c, where):
    """The case's per-step inputs on the device or in pinned host memory (pools stay on the device)."""
    out = dict(c)
    for name in _HOST:
        out[name] = c[name].to(DEV) if where == "device" else c[name].contiguous().pin_memory()
    return out


def _out(c, where):
    shape = c["q"].shape
    return (torch.empty(shape, dtype=torch.bfloat16, device=DEV) if where == "device"
            else torch.empty(shape, dtype=torch.bfloat16).pin_memory())


@pytest.mark.parametrize("d,hq,hkv", [(128, 32, 8), (64, 8, 2), (128, 12, 2)])
def test_append_decode_with_host_inputs_and_out(d, hq, hkv):
    lens = [300, 1, 0, 47, 1100]
    c = _case(lens, hq, hkv, d, seed=d + hq)
    res = {}
    for where in ("device", "host"):
        p = _placed(c, where)
        p["k_cache"], p["v_cache"] = c["k_cache"].clone(), c["v_cache"].clone()
        out = _out(c, where)
        err = pkv.new_error_word(DEV)
        pkv.paged_decode_attention_append(p["q"], p["k_cache"], p["v_cache"], p["k_new"], p["v_new"],
                                          p["block_tables"], p["context_lens"], c["scale"], out=out,
                                          error_word=err)
        torch.cuda.synchronize()
        assert pkv.read_error(err) == 0
        res[where] = (out.cpu(), p["k_cache"], p["v_cache"])
    assert torch.equal(bits_t(res["host"][0]), bits_t(res["device"][0]))
    assert torch.equal(res["host"][1], res["device"][1]) and torch.equal(res["host"][2], res["device"][2])
    # and against the oracle over the appended pools
    ref = oracle.paged_decode(bits(c["q"]), bits(res["host"][1]), bits(res["host"][2]), c["block_tables"].numpy(),
                              c["context_lens"].numpy(), c["scale"])
    assert_attn_close(res["host"][0], ref, f"host inputs d={d} hq={hq} hkv={hkv}")


def bits_t(t):
    return t.view(torch.int16)


def test_int8_append_decode_with_host_inputs():
    lens = [700, 33, 1]
    B, hq, hkv, d = 3, 16, 4, 128
    c = _case(lens, hq, hkv, d, seed=7)
    kq, ks = oracle.quantize_rows(bits(c["k_cache"].cpu()))
    vq, vs = oracle.quantize_rows(bits(c["v_cache"].cpu()))
    res = {}
    for where in ("device", "host"):
        p = _placed(c, where)
        pools = [torch.from_numpy(a.copy()).to(DEV) for a in (kq, vq, ks, vs)]
        out = _out(c, where)
        pkv.paged_decode_attention_append_q8(p["q"], *pools, p["k_new"], p["v_new"], p["block_tables"],
                                             p["context_lens"], c["scale"], out=out)
        torch.cuda.synchronize()
        res[where] = (out.cpu(), [t.cpu() for t in pools])
    assert torch.equal(bits_t(res["host"][0]), bits_t(res["device"][0]))
    for a, b in zip(res["host"][1], res["device"][1]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("window", [0, 40])
def test_plain_decode_host_inputs_device_out(window):
    c = _case([900, 64, 17, 0], 16, 4, 128, seed=11 + window)
    outs = []
    for where in ("device", "host"):
        p = _placed(c, where)
        outs.append(pkv.paged_decode_attention(p["q"], c["k_cache"], c["v_cache"], p["block_tables"],
                                               p["context_lens"], c["scale"], window))
    torch.cuda.synchronize()
    assert outs[0].is_cuda and outs[1].is_cuda
    assert torch.equal(bits_t(outs[0]), bits_t(outs[1]))


def test_sparse_gather_with_host_inputs():
    lens = [500, 90, 1200]
    B, hq, hkv, d, K = 3, 8, 2, 128, 96
    c = _case(lens, hq, hkv, d, seed=13)
    rng = np.random.default_rng(13)
    kept = np.full((B, hkv, K), -1, dtype=np.int32)
    kl = np.minimum(np.array(lens), K).astype(np.int32)
    for b in range(B):
        for g in range(hkv):
            kept[b, g, :kl[b]] = np.sort(rng.choice(lens[b], size=kl[b], replace=False))
    kept_d, kl_d = torch.from_numpy(kept).to(DEV), torch.from_numpy(kl).to(DEV)
    outs = []
    for where in ("device", "host"):
        p = _placed(c, where)
        outs.append(pkv.sparse_decode_attention(p["q"], c["k_cache"], c["v_cache"], p["block_tables"],
                                                p["context_lens"], kept_d, kl_d, c["scale"], out=_out(c, where)))
    torch.cuda.synchronize()
    assert torch.equal(bits_t(outs[0].cpu()), bits_t(outs[1].cpu()))


def test_flagged_host_input_steps_in_a_graph():
    """Steps over four pool copies, each reading its own pinned inputs and writing its own pinned
    output, declaring their inputs ready, captured in a CUDA graph: equal to eager device-input
    calls."""
    lens = [400, 1000, 3]
    cases = [_case(lens, 8, 2, 128, seed=20 + i) for i in range(4)]
    ws = torch.zeros(pkv.decode_workspace_bytes(3, 8, 2, 128, cases[0]["k_cache"].shape[0],
                                                cases[0]["block_tables"].shape[1]), dtype=torch.uint8, device=DEV)
    host = [_placed(c, "host") for c in cases]
    outs = [_out(c, "host") for c in cases]
    pools = [(c["k_cache"].clone(), c["v_cache"].clone()) for c in cases]
    s = torch.cuda.Stream(DEV)
    with torch.cuda.stream(s):
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            for h, o, (kc, vc) in zip(host, outs, pools):
                pkv.paged_decode_attention_append(h["q"], kc, vc, h["k_new"], h["v_new"], h["block_tables"],
                                                  h["context_lens"], h["scale"], out=o, workspace=ws,
                                                  inputs_ready=True, stream=s)
        gr.replay()
        torch.cuda.synchronize()
    for c, o, (kc, vc) in zip(cases, outs, pools):
        d = _placed(c, "device")
        k2, v2 = c["k_cache"].clone(), c["v_cache"].clone()
        ref = pkv.paged_decode_attention_append(d["q"], k2, v2, d["k_new"], d["v_new"], d["block_tables"],
                                                d["context_lens"], c["scale"])
        torch.cuda.synchronize()
        assert torch.equal(bits_t(o), bits_t(ref.cpu()))
        assert torch.equal(kc, k2) and torch.equal(vc, v2)


def test_pageable_host_memory_refused():
    c = _case([40, 8], 8, 2, 64, seed=3)
    with pytest.raises(ValueError, match="pinned host memory"):
        pkv.paged_decode_attention(c["q"], c["k_cache"], c["v_cache"], c["block_tables"].to(DEV),
                                   c["context_lens"].to(DEV), c["scale"])
    lib = pkv.load()
    import ctypes
    d = ctypes.c_void_p()
    buf = ctypes.create_string_buffer(64)
    assert lib.pkv_device_alias(ctypes.cast(buf, ctypes.c_void_p), ctypes.byref(d)) == \
        pkv.header_constants()["PKV_ERR_ARGUMENT"]
    assert d.value is None


def test_fixed_scratch_with_host_inputs():
    """The no-workspace entry point with pinned host inputs: out allocated on the device when not
    given, or a pinned host out; both equal to the device-input call bit for bit."""
    c = _case([600, 33, 1], 16, 4, 128, seed=17)
    d, h = _placed(c, "device"), _placed(c, "host")
    ref = pkv.paged_decode_attention_fixed_scratch(d["q"], c["k_cache"], c["v_cache"], d["block_tables"],
                                                   d["context_lens"], c["scale"])
    got = pkv.paged_decode_attention_fixed_scratch(h["q"], c["k_cache"], c["v_cache"], h["block_tables"],
                                                   h["context_lens"], c["scale"])
    got_h = pkv.paged_decode_attention_fixed_scratch(h["q"], c["k_cache"], c["v_cache"], h["block_tables"],
                                                     h["context_lens"], c["scale"], out=_out(c, "host"))
    torch.cuda.synchronize()
    assert got.is_cuda and not got_h.is_cuda
    assert torch.equal(bits_t(got), bits_t(ref)) and torch.equal(bits_t(got_h), bits_t(ref.cpu()))
