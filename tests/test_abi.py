"""The C-ABI library builds, loads and exports every entry point include/pkv.h declares; host
validation rejects bad arguments before anything touches a device.  No compute calls: these
run on a machine without a GPU."""
import ctypes
import subprocess

import pytest

from paged_kv_cache_mapped_gb300 import _build, _lib


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return _lib.load()


def _dims(B=4, hq=32, hkv=8, d=128, bs=16, nb=1000, mb=64):
    return _lib.PkvDims(B, hq, hkv, d, bs, nb, mb)


def test_every_declared_symbol_is_exported(lib):
    declared = _lib.header_functions()
    assert len(declared) == 23
    nm = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True)
    exported = {line.split()[-1] for line in nm.stdout.splitlines() if " T " in line}
    for name in declared:
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings(lib):
    c = _lib.header_constants()
    assert lib.pkv_status_string(c["PKV_OK"]) == b"ok"
    for name, val in c.items():
        if name.startswith("PKV_ERR_") and name != "PKV_ERR_CUDA_BASE":
            assert lib.pkv_status_string(val) not in (b"ok", b"unknown status"), name
        if name.startswith("PKV_DEV_") and val != 0:
            assert lib.pkv_device_error_string(val) != b"unknown device error", name


def test_workspace_queries(lib):
    d = _dims()
    n = lib.pkv_decode_workspace_bytes(ctypes.byref(d))
    # two partial slots of G heads x (d + 2) floats for each of 2048 static ranges and up to
    # three tail chunks per slice, whatever the context length
    assert n >= 2 * 2048 * 4 * 4 * (128 + 2) * 4 and n % 256 == 0
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(_dims(mb=8192))) == n
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(_dims(B=64))) >= n
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(_dims(hq=64))) > n      # G = 8
    assert lib.pkv_sparse_decode_workspace_bytes(ctypes.byref(d), 1540) == n
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(_dims(bs=32))) == 0
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(_dims(d=96))) == 0
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(_dims(hq=30))) == 0
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(_dims(hq=32, hkv=2))) == 0  # G = 16
    assert lib.pkv_sparse_decode_workspace_bytes(ctypes.byref(d), 0) == 0


def _decode(lib, dims, ptr=0x10000, ws_bytes=1 << 30, ws=0x20000, flags=0):
    P = ctypes.c_void_p
    return lib.pkv_paged_decode_attention(P(ptr), P(ptr), P(ptr), P(ptr), P(ptr), P(ptr),
                                          ctypes.c_float(0.1), 0, P(ws), ws_bytes,
                                          ctypes.byref(dims), flags, None, None)


def test_host_validation_codes(lib):
    c = _lib.header_constants()
    P = ctypes.c_void_p
    assert lib.pkv_paged_decode_attention(None, None, None, None, None, None, ctypes.c_float(1.0), 0,
                                          None, 0, None, 0, None, None) == c["PKV_ERR_NULL_POINTER"]
    assert _decode(lib, _dims(bs=8)) == c["PKV_ERR_BLOCK_SIZE"]
    assert _decode(lib, _dims(d=80)) == c["PKV_ERR_HEAD_DIM"]
    assert _decode(lib, _dims(hq=12, hkv=8)) == c["PKV_ERR_GQA"]
    assert _decode(lib, _dims(hq=32, hkv=2)) == c["PKV_ERR_GQA"]      # G = 16 exceeds one fragment
    assert _decode(lib, _dims(B=-1)) == c["PKV_ERR_DIMS"]
    assert _decode(lib, _dims(), ptr=0x10004) == c["PKV_ERR_ALIGNMENT"]
    assert _decode(lib, _dims(), ws_bytes=16) == c["PKV_ERR_WORKSPACE"]
    assert _decode(lib, _dims(), ws=0) == c["PKV_ERR_WORKSPACE"]
    assert _decode(lib, _dims(B=0)) == c["PKV_OK"]                    # empty batch: nothing to do
    assert _decode(lib, _dims(), flags=2) == c["PKV_ERR_ARGUMENT"]     # unknown flag bit
    assert _decode(lib, _dims(B=0), flags=c["PKV_DECODE_INPUTS_READY"]) == c["PKV_OK"]
    # append
    assert lib.pkv_kv_append(P(0x1000), P(0x1000), P(0x1000), P(0x1000), P(0x1000), -1,
                             ctypes.byref(_dims()), None, None) == c["PKV_ERR_DIMS"]
    assert lib.pkv_kv_append(P(0x1000), P(0x1000), P(0x1000), P(0x1000), P(0x1000), 0,
                             ctypes.byref(_dims()), None, None) == c["PKV_OK"]
    assert lib.pkv_kv_append(None, P(0x1000), P(0x1000), P(0x1000), P(0x1000), 4,
                             ctypes.byref(_dims()), None, None) == c["PKV_ERR_NULL_POINTER"]
    # selection
    assert lib.pkv_kv_select_topk(P(0x1000), P(0x1000), P(0x1000), 100, P(0x1000), -1, 4, 4,
                                  ctypes.byref(_dims()), 0, None, None) == c["PKV_ERR_ARGUMENT"]
    # unknown flag bits are refused before anything else is looked at
    assert lib.pkv_kv_select_topk(P(0x1000), P(0x1000), P(0x1000), 100, P(0x1000), 4, 4, 4,
                                  ctypes.byref(_dims()), 2, None, None) == c["PKV_ERR_ARGUMENT"]
    # score-emitting decode
    def scores(lse=0x30000, acc=0x40000, logits=0x50000, stride=64, k_new=None, v_new=None):
        return lib.pkv_paged_decode_attention_scores(
            P(0x10000), P(lse), P(acc), P(logits), stride, P(0x10000), P(0x10000), P(0x10000),
            P(k_new), P(v_new), P(0x10000), P(0x10000), ctypes.c_float(0.1), 0, P(0x20000), 16,
            ctypes.byref(_dims()), 0, None, None)
    assert scores(lse=0) == c["PKV_ERR_NULL_POINTER"]
    assert scores(stride=0) == c["PKV_ERR_DIMS"]
    assert scores(acc=0x40002) == c["PKV_ERR_ALIGNMENT"]
    assert scores(k_new=0x60000) == c["PKV_ERR_NULL_POINTER"]        # k_new without v_new
    assert scores() == c["PKV_ERR_WORKSPACE"]                         # 16-byte workspace
    # rolling admission
    def admit(cap=60, n_sink=4, n_recent=32, slot_pos=0x30000, dims=None, flags=0):
        return lib.pkv_kv_rolling_admit(P(0x10000), P(0x10000), P(0x10000), P(slot_pos), P(0x40000),
                                        P(0x50000), P(0x60000), P(0x70000), P(0x80000), cap, n_sink,
                                        n_recent, ctypes.byref(dims or _dims()), flags, None, None)
    assert admit(cap=0) == c["PKV_ERR_ARGUMENT"]
    assert admit(n_sink=40, n_recent=32) == c["PKV_ERR_ARGUMENT"]     # sinks + recent > capacity
    assert admit(cap=64 * 16 + 1) == c["PKV_ERR_DIMS"]                # more slots than the tables
    assert admit(slot_pos=0) == c["PKV_ERR_NULL_POINTER"]
    assert admit(dims=_dims(B=0)) == c["PKV_OK"]
    assert admit(dims=_dims(B=0), flags=c["PKV_ADMIT_INPUTS_READY"]) == c["PKV_OK"]
    assert admit(flags=2) == c["PKV_ERR_ARGUMENT"]                     # unknown flag bit
    # INT8 pools
    def q8_append(ks=0x30000, n=4):
        return lib.pkv_kv_append_q8(P(0x10000), P(0x10000), P(ks), P(0x40000), P(0x10000), P(0x10000),
                                    P(0x50000), n, ctypes.byref(_dims()), None, None)
    assert q8_append(n=0) == c["PKV_OK"]
    assert q8_append(n=-1) == c["PKV_ERR_DIMS"]
    assert q8_append(ks=0) == c["PKV_ERR_NULL_POINTER"]
    assert q8_append(ks=0x30004) == c["PKV_ERR_ALIGNMENT"]

    def q8_decode(vs=0x40000, ws_bytes=16, dims=None):
        return lib.pkv_paged_decode_attention_q8(P(0x10000), P(0x10000), P(0x10000), P(0x10000), P(0x30000),
                                                 P(vs), P(0x10000), P(0x10000), ctypes.c_float(0.1), 0,
                                                 P(0x20000), ws_bytes, ctypes.byref(dims or _dims()), 0, None,
                                                 None)
    assert q8_decode(vs=0) == c["PKV_ERR_NULL_POINTER"]
    assert q8_decode(vs=0x40008) == c["PKV_ERR_ALIGNMENT"]
    assert q8_decode() == c["PKV_ERR_WORKSPACE"]                      # 16-byte workspace
    assert q8_decode(dims=_dims(d=80)) == c["PKV_ERR_HEAD_DIM"]
    assert q8_decode(dims=_dims(B=0)) == c["PKV_OK"]
    def q8_scores(lse=0x50000, vs=0x40000, stride=64, dims=None):
        return lib.pkv_paged_decode_attention_scores_q8(
            P(0x10000), P(lse), P(0x60000), P(0x70000), stride, P(0x10000), P(0x10000), P(0x10000), P(0x30000),
            P(vs), P(0x10000), P(0x10000), ctypes.c_float(0.1), 0, P(0x20000), 16, ctypes.byref(dims or _dims()),
            0, None, None)
    assert q8_scores(lse=0) == c["PKV_ERR_NULL_POINTER"]
    assert q8_scores(vs=0x40008) == c["PKV_ERR_ALIGNMENT"]
    assert q8_scores(stride=0) == c["PKV_ERR_DIMS"]
    assert q8_scores() == c["PKV_ERR_WORKSPACE"]                     # 16-byte workspace
    assert q8_scores(dims=_dims(B=0)) == c["PKV_OK"]

    def q8_append_decode(kn=0x50000, dims=None):
        return lib.pkv_paged_decode_attention_append_q8(
            P(0x10000), P(0x10000), P(0x10000), P(0x10000), P(0x30000), P(0x40000), P(kn), P(0x60000),
            P(0x10000), P(0x10000), ctypes.c_float(0.1), 0, P(0x20000), 16, ctypes.byref(dims or _dims()), 0, None,
            None)
    assert q8_append_decode(kn=0) == c["PKV_ERR_NULL_POINTER"]
    assert q8_append_decode(kn=0x50008) == c["PKV_ERR_ALIGNMENT"]
    assert q8_append_decode() == c["PKV_ERR_WORKSPACE"]                # 16-byte workspace

    def q8_sparse(vs=0x40000, kept=0x50000, dims=None):
        return lib.pkv_sparse_decode_attention_q8(
            P(0x10000), P(0x10000), P(0x10000), P(0x10000), P(0x30000), P(vs), P(0x10000), P(0x10000), P(kept),
            P(0x60000), 16, ctypes.c_float(0.1), P(0x20000), 16, ctypes.byref(dims or _dims()), 0, None, None)
    assert q8_sparse(kept=0) == c["PKV_ERR_NULL_POINTER"]
    assert q8_sparse(vs=0x40008) == c["PKV_ERR_ALIGNMENT"]
    assert q8_sparse() == c["PKV_ERR_WORKSPACE"]                      # 16-byte workspace

    def q8_compact(dks=0x30000, max_kept=8, flags=0):
        return lib.pkv_kv_compact_q8(P(0x10000), P(0x10000), P(dks), P(0x40000), P(0x50000), 8, 4, P(0x10000),
                                     P(0x10000), P(0x30000), P(0x40000), P(0x50000), P(0x60000), P(0x70000),
                                     P(0x80000), max_kept, ctypes.byref(_dims()), flags, None, None)
    assert q8_compact(dks=0) == c["PKV_ERR_NULL_POINTER"]
    assert q8_compact(dks=0x30004) == c["PKV_ERR_ALIGNMENT"]
    assert q8_compact(max_kept=-1) == c["PKV_ERR_DIMS"]
    assert q8_compact(max_kept=0) == c["PKV_OK"]
    assert q8_compact(max_kept=0, flags=c["PKV_COMPACT_INPUTS_READY"]) == c["PKV_OK"]
    assert q8_compact(flags=2) == c["PKV_ERR_ARGUMENT"]                # unknown flag bit
    assert lib.pkv_kv_compact(P(0x10000), P(0x10000), P(0x50000), 8, 4, P(0x10000), P(0x10000), P(0x50000),
                              P(0x60000), P(0x70000), P(0x80000), 8, ctypes.byref(_dims()), 4, None,
                              None) == c["PKV_ERR_ARGUMENT"]

    def q8_admit(cap=60, n_sink=4, n_recent=32, ks=0x30000, flags=0):
        return lib.pkv_kv_rolling_admit_q8(P(0x10000), P(0x10000), P(ks), P(0x40000), P(0x10000), P(0x30000),
                                           P(0x40000), P(0x50000), P(0x60000), P(0x70000), P(0x80000), cap,
                                           n_sink, n_recent, ctypes.byref(_dims()), flags, None, None)
    assert q8_admit(cap=0) == c["PKV_ERR_ARGUMENT"]
    assert q8_admit(cap=64 * 16 + 1) == c["PKV_ERR_DIMS"]
    assert q8_admit(ks=0) == c["PKV_ERR_NULL_POINTER"]
    assert q8_admit(ks=0x30004) == c["PKV_ERR_ALIGNMENT"]
    assert q8_admit(flags=4) == c["PKV_ERR_ARGUMENT"]                  # unknown flag bit
    # prefill-window score
    def prefill(alpha=16, stride=64, lse=0x30000, qw=0x10000, dims=None):
        return lib.pkv_prefill_window_scores(P(0x40000), stride, P(lse), 0, P(qw), P(0x10000), P(0x10000),
                                             P(0x10000), alpha, ctypes.c_float(0.1), ctypes.byref(dims or _dims()),
                                             None, None)
    assert prefill(alpha=0) == c["PKV_ERR_ARGUMENT"]
    assert prefill(stride=0) == c["PKV_ERR_ARGUMENT"]
    assert prefill(alpha=4097) == c["PKV_ERR_DIMS"]                   # alpha * G above 16384
    assert prefill(lse=0) == c["PKV_ERR_NULL_POINTER"]
    assert prefill(qw=0x10008) == c["PKV_ERR_ALIGNMENT"]
    assert prefill(dims=_dims(hq=32, hkv=2)) == c["PKV_ERR_GQA"]
    assert prefill(dims=_dims(B=0)) == c["PKV_OK"]
    # sparse decode with no kept lists
    assert lib.pkv_sparse_decode_attention(P(0x10000), P(0x10000), P(0x10000), P(0x10000),
                                           P(0x10000), P(0x10000), None, None, 16,
                                           ctypes.c_float(0.1), P(0x20000), 1 << 30,
                                           ctypes.byref(_dims()), 0, None, None) == c["PKV_ERR_NULL_POINTER"]


def test_binding_rejects_cpu_tensors():
    import torch

    import paged_kv_cache_mapped_gb300 as pkv
    q = torch.zeros(2, 8, 64, dtype=torch.bfloat16)
    kc = torch.zeros(4, 8, 16, 64, dtype=torch.bfloat16)
    bt = torch.zeros(2, 2, dtype=torch.int32)
    lens = torch.ones(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        pkv.paged_decode_attention(q, kc, kc, bt, lens, 0.125)


def test_device_alias_refuses_null_and_unpinned_memory(lib):
    """pkv_device_alias: NULL arguments, and host memory that is not pinned (here: ordinary
    ctypes memory, or no device at all), come back as host errors with the output cleared; no
    device work is done."""
    c = _lib.header_constants()
    d = ctypes.c_void_p(0x1234)
    assert lib.pkv_device_alias(None, ctypes.byref(d)) == c["PKV_ERR_NULL_POINTER"]
    buf = ctypes.create_string_buffer(64)
    assert lib.pkv_device_alias(ctypes.cast(buf, ctypes.c_void_p), None) == c["PKV_ERR_NULL_POINTER"]
    assert lib.pkv_device_alias(ctypes.cast(buf, ctypes.c_void_p), ctypes.byref(d)) == c["PKV_ERR_ARGUMENT"]
    assert d.value is None
