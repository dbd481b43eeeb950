"""fp64 CPU oracle for the paged KV-cache decode path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg (and its
``--impl reference`` arm) may import this package.  The library under
``paged_kv_cache_mapped_gb300`` never does, and shares no code with it: the arithmetic
lives in ``pkv_oracle.c`` (plain C, fp64), this module only compiles it with gcc and
marshals numpy arrays through ctypes.

bf16 tensors are passed as their raw bits (numpy ``uint16``).  Every function raises
``OracleError`` when the C side refuses its input.

Parity status of each function (what pins it; see ``tests/test_oracle_*.py``):
  kv_cache_bytes   -- pinned by the worked examples of the KV-cache primer page (golden file)
  kv_append        -- pinned by a brute-force dict-of-slots model and untouched-slot checks
  paged_decode     -- pinned by closed forms (q=0, one token, equal rows, two tokens, W=1),
                      block-permutation invariance and torch SDPA (fp64) on contiguous K/V
  sparse_decode    -- pinned by kept=all == paged, and gather == compact-then-paged
  select_topk      -- pinned by a hand-worked golden case, exhaustive subset search on tiny
                      inputs and the selection invariants
  compact          -- pinned by a brute-force dict-of-slots model
  quantize_rows    -- pinned by exact round trips of codes times power-of-two scales, hand-worked
                      half-way ties, the rounding bound and the absmax element's code
  kv_append_q8     -- pinned by a dict-of-slots model over quantize_rows
  paged_decode_q8  -- pinned by equality with paged_decode where code * scale is a bf16 value,
                      and by torch SDPA (fp64) on the dequantized contiguous K/V
  sparse_decode_q8 -- pinned by equality with sparse_decode where code * scale is a bf16 value,
                      and kept = all == paged_decode_q8
  decode_scores_q8 -- pinned by equality with decode_scores where code * scale is a bf16 value,
                      and by torch softmax (fp64) on the dequantized K
  compact_q8       -- pinned by a dict-of-slots model (codes and row scales move together) and
                      by dequantize-then-compact == compact-then-dequantize
  rolling_admit_q8 -- pinned by the bf16 rolling admission's slot choice on the same scores and
                      by quantize_rows of the admitted rows
  prefill_scores   -- pinned by torch causal softmax (fp64), a segment's scores summing to G per
                      window row, the q = 0 closed form, alpha = 1 against decode_scores, the
                      given-lse property and block-permutation invariance
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    pass


_CODES = {
    -1: "invalid argument",
    -2: "slot outside the pool",
    -3: "block id outside the pool",
    -4: "token index outside the context / not ascending",
    -5: "invalid length",
    -6: "NaN score",
    -7: "out of memory",
    -8: "non-finite value",
}


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c into liboracle.so (with OpenMP when gcc supports it)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_num_threads.restype = i32
            lib.oracle_kv_cache_bytes.restype = i64
            lib.oracle_kv_cache_bytes.argtypes = [i64] * 6
            lib.oracle_kv_append.argtypes = [P, P, P, P, P, i64, i32, i32, i64]
            lib.oracle_paged_decode.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i64, i32,
                                                f64, i32, P, i64]
            lib.oracle_sparse_decode.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                                 i64, i32, f64, P, i64]
            lib.oracle_select_topk.argtypes = [P, P, P, i32, P, i32, i32, i32, i32, i32]
            lib.oracle_decode_scores.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i64, i32,
                                                 f64, i32, i64, P, i64]
            lib.oracle_rolling_admit.argtypes = [P, P, P, i64, i32, P, P, P, P, P, P, i32, i32, i32,
                                                 i32, i32, i32]
            lib.oracle_compact.argtypes = [P, P, P, i64, i32, P, P, P, P, P, P, i32, i32, i32,
                                           i32, i64, i32]
            lib.oracle_prefill_scores.argtypes = [P, P, i32, P, P, P, P, i32, i32, i32, i32, i64, i32,
                                                  i32, f64, i64, P, i64]
            lib.oracle_quantize_rows.argtypes = [P, P, P, i64, i32]
            lib.oracle_kv_append_q8.argtypes = [P, P, P, P, P, P, P, i64, i32, i32, i64]
            lib.oracle_paged_decode_q8.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i64,
                                                   i32, f64, i32, P, i64]
            lib.oracle_decode_scores_q8.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i64, i32,
                                                    f64, i32, i64, P, i64]
            lib.oracle_compact_q8.argtypes = [P, P, P, P, P, i64, i32, P, P, P, P, P, P, P, P, i32, i32,
                                              i32, i32, i64, i32]
            lib.oracle_rolling_admit_q8.argtypes = [P, P, P, P, P, i64, i32, P, P, P, P, P, P, i32, i32,
                                                    i32, i32, i32, i32]
            lib.oracle_sparse_decode_q8.argtypes = [P, P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                                    i64, i32, f64, P, i64]
            for name in ("oracle_sparse_decode_q8", "oracle_kv_append", "oracle_paged_decode", "oracle_sparse_decode",
                         "oracle_select_topk", "oracle_compact", "oracle_decode_scores",
                         "oracle_rolling_admit", "oracle_quantize_rows", "oracle_kv_append_q8",
                         "oracle_paged_decode_q8", "oracle_prefill_scores", "oracle_decode_scores_q8",
                         "oracle_compact_q8", "oracle_rolling_admit_q8"):
                getattr(lib, name).restype = i32
            _lib = lib
    return _lib


def _check(status: int, what: str) -> None:
    if status != 0:
        raise OracleError(f"{what}: {_CODES.get(status, status)}")


def _arr(x, dtype) -> np.ndarray:
    a = np.ascontiguousarray(x)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads the oracle's parallel loops use from now on (timing only; results do not depend on it)."""
    lib = _load()
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_num_threads.restype = None
    lib.oracle_set_num_threads(int(n))


def kv_cache_bytes(batch, layers, heads, head_dim, seq_len, dtype_bytes) -> int:
    return int(_load().oracle_kv_cache_bytes(batch, layers, heads, head_dim, seq_len, dtype_bytes))


def kv_append(k_cache, v_cache, k, v, slot_mapping):
    """Return copies of the uint16 pools [NB,Hkv,16,d] after writing k, v [T,Hkv,d] at the slots."""
    kc = np.array(_arr(k_cache, np.uint16), copy=True)
    vc = np.array(_arr(v_cache, np.uint16), copy=True)
    k = _arr(k, np.uint16)
    v = _arr(v, np.uint16)
    slots = _arr(slot_mapping, np.int64)
    nb, hkv, bs, d = kc.shape
    assert bs == 16 and k.shape == (slots.shape[0], hkv, d) and v.shape == k.shape
    _check(_load().oracle_kv_append(_ptr(kc), _ptr(vc), _ptr(k), _ptr(v), _ptr(slots),
                                    slots.shape[0], hkv, d, nb), "kv_append")
    return kc, vc


def _rows(rows, batch, hq):
    if rows is None:
        return None, batch * hq
    r = _arr(np.asarray(rows, dtype=np.int64), np.int64)
    return r, r.shape[0]


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale, window=0, rows=None):
    """fp64 attention.  rows=None -> [B,Hq,d]; else a list of b*Hq+h -> [len(rows), d]."""
    q = _arr(q, np.uint16)
    kc = _arr(k_cache, np.uint16)
    vc = _arr(v_cache, np.uint16)
    bt = _arr(block_tables, np.int32)
    lens = _arr(context_lens, np.int32)
    b, hq, d = q.shape
    nb, hkv, bs, d2 = kc.shape
    assert bs == 16 and d2 == d and vc.shape == kc.shape and bt.shape[0] == b
    r, n = _rows(rows, b, hq)
    out = np.zeros((n, d), dtype=np.float64)
    _check(_load().oracle_paged_decode(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(lens),
                                       b, hq, hkv, d, nb, bt.shape[1], float(scale), int(window),
                                       None if r is None else _ptr(r), n), "paged_decode")
    return out.reshape(b, hq, d) if rows is None else out


def sparse_decode(q, k_cache, v_cache, block_tables, context_lens, kept, kept_lens, scale, rows=None):
    """fp64 attention over kept[b][g][:kept_lens[b]]."""
    q = _arr(q, np.uint16)
    kc = _arr(k_cache, np.uint16)
    vc = _arr(v_cache, np.uint16)
    bt = _arr(block_tables, np.int32)
    lens = _arr(context_lens, np.int32)
    kept = _arr(kept, np.int32)
    kl = _arr(kept_lens, np.int32)
    b, hq, d = q.shape
    nb, hkv, bs, _ = kc.shape
    assert kept.shape[:2] == (b, hkv)
    r, n = _rows(rows, b, hq)
    out = np.zeros((n, d), dtype=np.float64)
    _check(_load().oracle_sparse_decode(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(lens),
                                        _ptr(kept), _ptr(kl), kept.shape[2], b, hq, hkv, d, nb,
                                        bt.shape[1], float(scale), None if r is None else _ptr(r), n),
           "sparse_decode")
    return out.reshape(b, hq, d) if rows is None else out


def decode_scores(q, k_cache, block_tables, context_lens, scale, window=0, stride=None, segs=None):
    """fp64 sparsification score of one decode step and the rows' log-sum-exp.

    segs=None -> (score_add [B, Hkv, stride], lse [B, Hq]); else a list of b*Hkv+g ->
    (score_add [len(segs), stride], lse [len(segs), G]).  stride defaults to max L_b."""
    q = _arr(q, np.uint16)
    kc = _arr(k_cache, np.uint16)
    bt = _arr(block_tables, np.int32)
    lens = _arr(context_lens, np.int32)
    b, hq, d = q.shape
    nb, hkv, bs, d2 = kc.shape
    assert bs == 16 and d2 == d and bt.shape[0] == b
    g = hq // hkv
    if stride is None:
        stride = max(int(lens.max()) if lens.size else 0, 1)
    if segs is None:
        s_arr, n = None, b * hkv
    else:
        s_arr = _arr(np.asarray(segs, dtype=np.int64), np.int64)
        n = s_arr.shape[0]
    score = np.zeros((n, stride), dtype=np.float64)
    lse = np.zeros((n, g), dtype=np.float64)
    _check(_load().oracle_decode_scores(_ptr(score), _ptr(lse), _ptr(q), _ptr(kc), _ptr(bt), _ptr(lens),
                                        b, hq, hkv, d, nb, bt.shape[1], float(scale), int(window),
                                        int(stride), None if s_arr is None else _ptr(s_arr), n),
           "decode_scores")
    if segs is None:
        return score.reshape(b, hkv, stride), lse.reshape(b, hq)
    return score, lse


def select_topk(scores, context_lens, n_sink, n_recent, k_top):
    """Return (kept [B,Hkv,K] int32 with -1 past kept_lens, kept_lens [B])."""
    s = _arr(scores, np.float32)
    lens = _arr(context_lens, np.int32)
    b, hkv, stride = s.shape
    kmax = n_sink + k_top + n_recent
    kept = np.full((b, hkv, kmax), -1, dtype=np.int32)
    kl = np.zeros((b,), dtype=np.int32)
    _check(_load().oracle_select_topk(_ptr(kept), _ptr(kl), _ptr(s), stride, _ptr(lens), b, hkv,
                                      n_sink, n_recent, k_top), "select_topk")
    return kept, kl


def compact(dst_k, dst_v, dst_block_tables, src_k, src_v, src_block_tables, context_lens, kept,
            kept_lens):
    """Return copies of the destination pools after the compaction copy."""
    dk = np.array(_arr(dst_k, np.uint16), copy=True)
    dv = np.array(_arr(dst_v, np.uint16), copy=True)
    dbt = _arr(dst_block_tables, np.int32)
    sk = _arr(src_k, np.uint16)
    sv = _arr(src_v, np.uint16)
    sbt = _arr(src_block_tables, np.int32)
    lens = _arr(context_lens, np.int32)
    kept = _arr(kept, np.int32)
    kl = _arr(kept_lens, np.int32)
    b, hkv, max_kept = kept.shape
    d = sk.shape[3]
    _check(_load().oracle_compact(_ptr(dk), _ptr(dv), _ptr(dbt), dk.shape[0], dbt.shape[1],
                                  _ptr(sk), _ptr(sv), _ptr(sbt), _ptr(lens), _ptr(kept), _ptr(kl),
                                  max_kept, b, hkv, d, sk.shape[0], sbt.shape[1]), "compact")
    return dk, dv


def rolling_admit(k_cache, v_cache, block_tables, slot_pos, slot_score, kept_lens, context_lens, k_new, v_new,
                  n_sink, n_recent):
    """One step's rolling admission; returns updated copies (k_cache, v_cache, slot_pos,
    slot_score, kept_lens).  slot_pos/slot_score are [B, Hkv, capacity]."""
    kc = np.array(_arr(k_cache, np.uint16), copy=True)
    vc = np.array(_arr(v_cache, np.uint16), copy=True)
    bt = _arr(block_tables, np.int32)
    pos = np.array(_arr(slot_pos, np.int32), copy=True)
    sc = np.array(_arr(slot_score, np.float32), copy=True)
    kl = np.array(_arr(kept_lens, np.int32), copy=True)
    lens = _arr(context_lens, np.int32)
    kn = _arr(k_new, np.uint16)
    vn = _arr(v_new, np.uint16)
    nb, hkv, bs, d = kc.shape
    b, hkv2, cap = pos.shape
    assert bs == 16 and hkv2 == hkv and sc.shape == pos.shape and kn.shape == (b, hkv, d)
    _check(_load().oracle_rolling_admit(_ptr(kc), _ptr(vc), _ptr(bt), nb, bt.shape[1], _ptr(pos), _ptr(sc),
                                        _ptr(kl), _ptr(lens), _ptr(kn), _ptr(vn), b, hkv, d, cap,
                                        int(n_sink), int(n_recent)), "rolling_admit")
    return kc, vc, pos, sc, kl


def quantize_rows(x):
    """INT8 quantization of the last axis of x (bf16 bits): (codes x.shape as stored, each code c as the
    byte c + 128 (uint8), scales fp32 x.shape[:-1])."""
    x = _arr(x, np.uint16)
    d = x.shape[-1]
    n = x.size // d if d else 0
    codes = np.zeros(x.shape, dtype=np.uint8)
    scales = np.zeros(x.shape[:-1], dtype=np.float32)
    _check(_load().oracle_quantize_rows(_ptr(codes), _ptr(scales), _ptr(x), n, d), "quantize_rows")
    return codes, scales


def kv_append_q8(k_codes, v_codes, k_scales, v_scales, k, v, slot_mapping):
    """Return copies of the INT8 pools ([NB,Hkv,16,d] uint8 codes c stored as c + 128, [NB,Hkv,16] fp32 scales)
    after quantizing k, v [T,Hkv,d] (bf16 bits) into the slots."""
    kc = np.array(_arr(k_codes, np.uint8), copy=True)
    vc = np.array(_arr(v_codes, np.uint8), copy=True)
    ks = np.array(_arr(k_scales, np.float32), copy=True)
    vs = np.array(_arr(v_scales, np.float32), copy=True)
    k = _arr(k, np.uint16)
    v = _arr(v, np.uint16)
    slots = _arr(slot_mapping, np.int64)
    nb, hkv, bs, d = kc.shape
    assert bs == 16 and vc.shape == kc.shape and ks.shape == (nb, hkv, 16) and vs.shape == ks.shape
    assert k.shape == (slots.shape[0], hkv, d) and v.shape == k.shape
    _check(_load().oracle_kv_append_q8(_ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(k), _ptr(v), _ptr(slots),
                                       slots.shape[0], hkv, d, nb), "kv_append_q8")
    return kc, vc, ks, vs


def paged_decode_q8(q, k_codes, k_scales, v_codes, v_scales, block_tables, context_lens, scale, window=0,
                    rows=None):
    """fp64 attention over INT8 pools (values code * scale).  Shapes as paged_decode."""
    q = _arr(q, np.uint16)
    kc = _arr(k_codes, np.uint8)
    vc = _arr(v_codes, np.uint8)
    ks = _arr(k_scales, np.float32)
    vs = _arr(v_scales, np.float32)
    bt = _arr(block_tables, np.int32)
    lens = _arr(context_lens, np.int32)
    b, hq, d = q.shape
    nb, hkv, bs, d2 = kc.shape
    assert bs == 16 and d2 == d and vc.shape == kc.shape and ks.shape == (nb, hkv, 16) and vs.shape == ks.shape
    assert bt.shape[0] == b
    r, n = _rows(rows, b, hq)
    out = np.zeros((n, d), dtype=np.float64)
    _check(_load().oracle_paged_decode_q8(_ptr(out), _ptr(q), _ptr(kc), _ptr(ks), _ptr(vc), _ptr(vs), _ptr(bt),
                                          _ptr(lens), b, hq, hkv, d, nb, bt.shape[1], float(scale), int(window),
                                          None if r is None else _ptr(r), n), "paged_decode_q8")
    return out.reshape(b, hq, d) if rows is None else out


def prefill_scores(q_win, k_cache, block_tables, context_lens, alpha, scale, lse=None, stride=None, segs=None):
    """fp64 prefill-window score.  q_win [B, alpha, Hq, d] (bf16 bits): row r is position
    L_b - alpha + r.  lse [B, Hq, alpha] given, or None to compute it.  Returns
    (score_add [B, Hkv, stride] or [len(segs), stride], lse [B, Hq, alpha])."""
    q = _arr(q_win, np.uint16)
    kc = _arr(k_cache, np.uint16)
    bt = _arr(block_tables, np.int32)
    lens = _arr(context_lens, np.int32)
    b, a, hq, d = q.shape
    nb, hkv, bs, d2 = kc.shape
    assert a == alpha and bs == 16 and d2 == d and bt.shape[0] == b
    if stride is None:
        stride = max(int(lens.max()) if lens.size else 0, 1)
    given = lse is not None
    lse_arr = np.array(lse, dtype=np.float64, copy=True) if given else np.zeros((b, hq, alpha), dtype=np.float64)
    assert lse_arr.shape == (b, hq, alpha)
    if segs is None:
        s_arr, n = None, b * hkv
    else:
        s_arr = _arr(np.asarray(segs, dtype=np.int64), np.int64)
        n = s_arr.shape[0]
    score = np.zeros((n, stride), dtype=np.float64)
    _check(_load().oracle_prefill_scores(_ptr(score), _ptr(lse_arr), int(given), _ptr(q), _ptr(kc), _ptr(bt),
                                         _ptr(lens), b, hq, hkv, d, nb, bt.shape[1], int(alpha), float(scale),
                                         int(stride), None if s_arr is None else _ptr(s_arr), n), "prefill_scores")
    if segs is None:
        score = score.reshape(b, hkv, stride)
    return score, lse_arr


def decode_scores_q8(q, k_codes, k_scales, block_tables, context_lens, scale, window=0, stride=None, segs=None):
    """decode_scores over an INT8 K pool (values code * scale); same returns."""
    q = _arr(q, np.uint16)
    kc = _arr(k_codes, np.uint8)
    ks = _arr(k_scales, np.float32)
    bt = _arr(block_tables, np.int32)
    lens = _arr(context_lens, np.int32)
    b, hq, d = q.shape
    nb, hkv, bs, d2 = kc.shape
    assert bs == 16 and d2 == d and ks.shape == (nb, hkv, 16) and bt.shape[0] == b
    g = hq // hkv
    if stride is None:
        stride = max(int(lens.max()) if lens.size else 0, 1)
    if segs is None:
        s_arr, n = None, b * hkv
    else:
        s_arr = _arr(np.asarray(segs, dtype=np.int64), np.int64)
        n = s_arr.shape[0]
    score = np.zeros((n, stride), dtype=np.float64)
    lse = np.zeros((n, g), dtype=np.float64)
    _check(_load().oracle_decode_scores_q8(_ptr(score), _ptr(lse), _ptr(q), _ptr(kc), _ptr(ks), _ptr(bt),
                                           _ptr(lens), b, hq, hkv, d, nb, bt.shape[1], float(scale), int(window),
                                           int(stride), None if s_arr is None else _ptr(s_arr), n),
           "decode_scores_q8")
    if segs is None:
        return score.reshape(b, hkv, stride), lse.reshape(b, hq)
    return score, lse


def compact_q8(dst_k, dst_v, dst_ks, dst_vs, dst_block_tables, src_k, src_v, src_ks, src_vs, src_block_tables,
               context_lens, kept, kept_lens):
    """INT8 compaction; returns copies (dst_k, dst_v, dst_ks, dst_vs) of the destination pools."""
    dk = np.array(_arr(dst_k, np.uint8), copy=True)
    dv = np.array(_arr(dst_v, np.uint8), copy=True)
    dks = np.array(_arr(dst_ks, np.float32), copy=True)
    dvs = np.array(_arr(dst_vs, np.float32), copy=True)
    dbt = _arr(dst_block_tables, np.int32)
    sk = _arr(src_k, np.uint8)
    sv = _arr(src_v, np.uint8)
    sks = _arr(src_ks, np.float32)
    svs = _arr(src_vs, np.float32)
    sbt = _arr(src_block_tables, np.int32)
    lens = _arr(context_lens, np.int32)
    kept = _arr(kept, np.int32)
    kl = _arr(kept_lens, np.int32)
    b, hkv, max_kept = kept.shape
    d = sk.shape[3]
    assert dks.shape == dk.shape[:3] and sks.shape == sk.shape[:3]
    _check(_load().oracle_compact_q8(_ptr(dk), _ptr(dv), _ptr(dks), _ptr(dvs), _ptr(dbt), dk.shape[0],
                                     dbt.shape[1], _ptr(sk), _ptr(sv), _ptr(sks), _ptr(svs), _ptr(sbt),
                                     _ptr(lens), _ptr(kept), _ptr(kl), max_kept, b, hkv, d, sk.shape[0],
                                     sbt.shape[1]), "compact_q8")
    return dk, dv, dks, dvs


def rolling_admit_q8(k_codes, v_codes, k_scales, v_scales, block_tables, slot_pos, slot_score, kept_lens,
                     context_lens, k_new, v_new, n_sink, n_recent):
    """rolling_admit into INT8 pools; returns updated copies (k_codes, v_codes, k_scales,
    v_scales, slot_pos, slot_score, kept_lens)."""
    kc = np.array(_arr(k_codes, np.uint8), copy=True)
    vc = np.array(_arr(v_codes, np.uint8), copy=True)
    ks = np.array(_arr(k_scales, np.float32), copy=True)
    vs = np.array(_arr(v_scales, np.float32), copy=True)
    bt = _arr(block_tables, np.int32)
    pos = np.array(_arr(slot_pos, np.int32), copy=True)
    sc = np.array(_arr(slot_score, np.float32), copy=True)
    kl = np.array(_arr(kept_lens, np.int32), copy=True)
    lens = _arr(context_lens, np.int32)
    kn = _arr(k_new, np.uint16)
    vn = _arr(v_new, np.uint16)
    nb, hkv, bs, d = kc.shape
    b, hkv2, cap = pos.shape
    assert bs == 16 and hkv2 == hkv and sc.shape == pos.shape and kn.shape == (b, hkv, d)
    assert ks.shape == (nb, hkv, 16) and vs.shape == ks.shape
    _check(_load().oracle_rolling_admit_q8(_ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt), nb, bt.shape[1],
                                           _ptr(pos), _ptr(sc), _ptr(kl), _ptr(lens), _ptr(kn), _ptr(vn), b, hkv,
                                           d, cap, int(n_sink), int(n_recent)), "rolling_admit_q8")
    return kc, vc, ks, vs, pos, sc, kl


def sparse_decode_q8(q, k_codes, k_scales, v_codes, v_scales, block_tables, context_lens, kept, kept_lens, scale,
                     rows=None):
    """sparse_decode over INT8 pools (values code * scale).  Shapes as sparse_decode."""
    q = _arr(q, np.uint16)
    kc = _arr(k_codes, np.uint8)
    vc = _arr(v_codes, np.uint8)
    ks = _arr(k_scales, np.float32)
    vs = _arr(v_scales, np.float32)
    bt = _arr(block_tables, np.int32)
    lens = _arr(context_lens, np.int32)
    kept = _arr(kept, np.int32)
    kl = _arr(kept_lens, np.int32)
    b, hq, d = q.shape
    nb, hkv, bs, _ = kc.shape
    assert bs == 16 and vc.shape == kc.shape and ks.shape == (nb, hkv, 16) and vs.shape == ks.shape
    assert kept.shape[:2] == (b, hkv)
    r, n = _rows(rows, b, hq)
    out = np.zeros((n, d), dtype=np.float64)
    _check(_load().oracle_sparse_decode_q8(_ptr(out), _ptr(q), _ptr(kc), _ptr(ks), _ptr(vc), _ptr(vs), _ptr(bt),
                                           _ptr(lens), _ptr(kept), _ptr(kl), kept.shape[2], b, hq, hkv, d, nb,
                                           bt.shape[1], float(scale), None if r is None else _ptr(r), n),
           "sparse_decode_q8")
    return out.reshape(b, hq, d) if rows is None else out
