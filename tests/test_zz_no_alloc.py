"""The allocation-free decode entry point (pkv_paged_decode_attention_fixed_scratch).

It serves callers that cannot allocate device memory -- a plain C program or plugin with no
device allocator of its own, or a host runtime that owns the device heap and forbids
cudaMalloc -- by keeping its split-K scratch in a fixed static device array inside the
library.  These tests call it through the C ABI (ctypes on libpkv.so, no Python helper in
between) twice in a row and compare both results with the fp64 oracle and with the
workspace-taking entry point, within the same tolerance the other attention tests use (the
llama8b-sized case on a sample of rows the oracle computes one by one).  They also check that
a shape whose partial results do not fit the fixed scratch (G = 8 at head_dim 128) is refused
without touching the device, and that the next call still works.  This file is collected last,
and each test builds its own inputs, so it passes alone in a fresh process as well as after the
other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_mapped_gb300 as pkv
from paged_kv_cache_mapped_gb300 import _lib
from paged_kv_cache_mapped_gb300 import inputs as W
from helpers import MAX_ABS, REL_L2, attn_errors, bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
C = _lib.header_constants()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _dims(case):
    q, kc, bt = case["q"], case["k_cache"], case["block_tables"]
    return _lib.PkvDims(q.shape[0], q.shape[1], kc.shape[1], kc.shape[3], 16, kc.shape[0], bt.shape[1])


def _fixed(case, out, window=0, err=None):
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    return _lib.load().pkv_paged_decode_attention_fixed_scratch(
        _p(out), _p(case["q"]), _p(case["k_cache"]), _p(case["v_cache"]), _p(case["block_tables"]),
        _p(case["context_lens"]), ctypes.c_float(case["scale"]), window, ctypes.byref(_dims(case)),
        None if err is None else _p(err), stream)


def _with_workspace(case, window=0):
    dims = _dims(case)
    lib = _lib.load()
    ws = torch.zeros(lib.pkv_decode_workspace_bytes(ctypes.byref(dims)), dtype=torch.uint8, device=DEV)
    out = torch.empty_like(case["q"])
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    st = lib.pkv_paged_decode_attention(
        _p(out), _p(case["q"]), _p(case["k_cache"]), _p(case["v_cache"]), _p(case["block_tables"]),
        _p(case["context_lens"]), ctypes.c_float(case["scale"]), window, _p(ws), ws.numel(),
        ctypes.byref(dims), 0, None, stream)
    assert st == C["PKV_OK"]
    return out


def _compare(got, ref, what):
    mx, rel = attn_errors(got, ref.double().cpu().numpy())
    assert torch.isfinite(got.float()).all(), what
    assert mx <= MAX_ABS and rel <= REL_L2, f"{what}: max-abs {mx:.3e} rel-L2 {rel:.3e}"


def _oracle_rows(case, rows, window):
    return oracle.paged_decode(bits(case["q"]), bits(case["k_cache"]), bits(case["v_cache"]),
                               case["block_tables"].cpu().numpy(), case["context_lens"].cpu().numpy(),
                               case["scale"], window, rows=rows)


def _rows(name, case):
    """Every row of the tiny case; for llama8b a fixed sample (each sequence's first and last
    query head plus 48 random rows)."""
    B, hq = case["q"].shape[:2]
    if name == "tiny":
        return list(range(B * hq))
    rng = np.random.default_rng(77)
    rows = {b * hq for b in range(B)} | {b * hq + hq - 1 for b in range(B)}
    rows |= set(rng.choice(B * hq, size=48, replace=False).tolist())
    return sorted(rows)


@pytest.mark.parametrize("name,window", [("tiny", 0), ("tiny", 50), ("llama8b", 0)])
def test_fixed_scratch_matches_oracle_and_workspace_entry_point_twice(name, window):
    case = W.make_layer(W.WORKLOADS[name], device=DEV, device_rng=(name != "tiny"))
    rows = _rows(name, case)
    idx = torch.tensor(rows, device=DEV)
    d = case["q"].shape[2]
    ref_oracle = torch.from_numpy(_oracle_rows(case, rows, window))
    ref_ws = _with_workspace(case, window).float().view(-1, d)[idx]
    err = pkv.new_error_word(DEV)
    for call in range(2):
        out = torch.full_like(case["q"], float("nan"))
        assert _fixed(case, out, window, err) == C["PKV_OK"]
        torch.cuda.synchronize()
        got = out.view(-1, d)[idx]
        _compare(got, ref_oracle, f"{name} window={window} call {call} against the oracle")
        _compare(got, ref_ws, f"{name} window={window} call {call} against the workspace entry point")
    assert pkv.read_error(err) == 0


def test_fixed_scratch_refuses_oversized_shapes():
    # G = 8 query heads per kv head at d = 128: the partials of 2048 worker ranges take
    # ~17 MB, more than the fixed scratch holds: refused, nothing run
    B, hq, hkv, d = 2, 64, 8, 128
    lens = torch.tensor([40, 17], dtype=torch.int32)
    wl = W.Workload("g8", 90, batch=B, num_q_heads=hq, num_kv_heads=hkv, head_dim=d)
    case = W.make_layer(wl, device=DEV, lengths=lens, num_blocks=8, max_blocks=4)
    need = _lib.load().pkv_decode_workspace_bytes(ctypes.byref(_dims(case)))
    assert need > C["PKV_FIXED_SCRATCH_BYTES"]
    out = torch.zeros_like(case["q"])
    err = pkv.new_error_word(DEV)
    assert _fixed(case, out, err=err) == C["PKV_ERR_WORKSPACE"]
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
    assert pkv.read_error(err) == 0
    # the refusal left the scratch usable: a normal call right after it is exact and clean
    tiny = W.make_layer(W.WORKLOADS["tiny"], device=DEV)
    out = torch.full_like(tiny["q"], float("nan"))
    assert _fixed(tiny, out, err=err) == C["PKV_OK"]
    torch.cuda.synchronize()
    assert pkv.read_error(err) == 0
    _compare(out, torch.from_numpy(_oracle_rows(tiny, None, 0)), "tiny call after a refused one")
