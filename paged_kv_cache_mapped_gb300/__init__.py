"""Paged KV-cache decode attention for GB300 (sm_103a).

Python binding of libpkv (declared in include/pkv.h).  Each function checks the torch
tensors it is given, builds the C shape record and calls the C-ABI entry point of the same
name (``pkv_<name>``) on the current CUDA stream.  All computation happens in the library's
CUDA kernels; CPU tensors are rejected, there is no fallback path.  PyTorch only provides
device memory (outputs ``torch.empty``, workspaces ``torch.zeros``, on the inputs' device) and the
stream handle.
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import PkvDims, PkvError, check, header_constants, header_functions, load

__all__ = [
    "BLOCK_SIZE", "PkvError", "kv_append", "decode_workspace_bytes", "paged_decode_attention",
    "sparse_decode_workspace_bytes", "sparse_decode_attention", "kv_select_topk", "kv_compact",
    "read_error", "new_error_word", "header_constants", "header_functions",
    "paged_decode_attention_fixed_scratch", "paged_decode_attention_append",
    "paged_decode_attention_scores", "kv_rolling_admit",
    "kv_append_q8",
    "paged_decode_attention_q8",
    "prefill_window_scores",
    "paged_decode_attention_scores_q8", "kv_compact_q8", "kv_rolling_admit_q8",
    "paged_decode_attention_append_q8", "sparse_decode_attention_q8",
]

BLOCK_SIZE = 16
_INPUTS_READY = header_constants()["PKV_DECODE_INPUTS_READY"]
_SELECT_READY = header_constants()["PKV_SELECT_INPUTS_READY"]
_COMPACT_READY = header_constants()["PKV_COMPACT_INPUTS_READY"]
_ADMIT_READY = header_constants()["PKV_ADMIT_INPUTS_READY"]


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:  # pinned host memory (admitted by _need): its device address
        base = t.untyped_storage().data_ptr()
        d = ctypes.c_void_p()
        check("pkv_device_alias", load().pkv_device_alias(ctypes.c_void_p(base), ctypes.byref(d)))
        return ctypes.c_void_p(d.value + (t.data_ptr() - base))
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, ndim, device=None, host_ok=False):
    """host_ok: the argument may also be pinned host memory, which the kernels reach in place."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    on_host = host_ok and not t.is_cuda and t.is_pinned()
    if not t.is_cuda and not on_host:
        where = "a CUDA device or pinned host memory" if host_ok else "a CUDA device"
        raise ValueError(f"{name} must live on {where} (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if device is not None and not on_host and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _pool_dims(k_cache, v_cache):
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4, k_cache.device)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    nb, hkv, bs, d = k_cache.shape
    if bs != BLOCK_SIZE:
        raise ValueError(f"pool block size must be {BLOCK_SIZE}")
    return nb, hkv, d


def _dims(batch, hq, hkv, d, nb, mb):
    return PkvDims(batch, hq, hkv, d, BLOCK_SIZE, nb, mb)


def new_error_word(device) -> torch.Tensor:
    """A zeroed device int32 the kernels report device-side errors into."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def read_error(error_word: torch.Tensor, clear: bool = False, stream=None) -> int:
    """Synchronise the stream and return the device error code (0 = none)."""
    _need(error_word, "error_word", torch.int32, 1)
    return int(load().pkv_read_error(_ptr(error_word), int(bool(clear)),
                                     _stream(stream, error_word.device)))


def kv_append(k_cache, v_cache, k, v, slot_mapping, *, error_word=None, stream=None):
    """Write k, v [T, Hkv, d] into the pools [NB, Hkv, 16, d] at slot_mapping [T] (int64)."""
    nb, hkv, d = _pool_dims(k_cache, v_cache)
    dev = k_cache.device
    _need(k, "k", torch.bfloat16, 3, dev)
    _need(v, "v", torch.bfloat16, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    T = slot_mapping.shape[0]
    if k.shape != (T, hkv, d) or v.shape != k.shape:
        raise ValueError("k/v must be [num_tokens, num_kv_heads, head_dim]")
    dims = _dims(0, 0, hkv, d, nb, 0)
    check("pkv_kv_append", load().pkv_kv_append(
        _ptr(k_cache), _ptr(v_cache), _ptr(k), _ptr(v), _ptr(slot_mapping), T, ctypes.byref(dims),
        _ptr(error_word), _stream(stream, dev)))


def _q8_pool_dims(k_codes, v_codes, k_scales, v_scales):
    _need(k_codes, "k_codes", torch.uint8, 4)
    dev = k_codes.device
    _need(v_codes, "v_codes", torch.uint8, 4, dev)
    _need(k_scales, "k_scales", torch.float32, 3, dev)
    _need(v_scales, "v_scales", torch.float32, 3, dev)
    if v_codes.shape != k_codes.shape:
        raise ValueError("k_codes and v_codes shapes differ")
    nb, hkv, bs, d = k_codes.shape
    if bs != BLOCK_SIZE:
        raise ValueError(f"pool block size must be {BLOCK_SIZE}")
    if k_scales.shape != (nb, hkv, BLOCK_SIZE) or v_scales.shape != k_scales.shape:
        raise ValueError("scale pools must be [num_blocks, num_kv_heads, 16]")
    return nb, hkv, d


def kv_append_q8(k_codes, v_codes, k_scales, v_scales, k, v, slot_mapping, *, error_word=None, stream=None):
    """Quantize k, v [T, Hkv, d] (bf16) into the INT8 pools at slot_mapping [T] (int64):
    codes [NB, Hkv, 16, d] uint8 (each code c stored as the byte c + 128) and one fp32 scale per
    row, [NB, Hkv, 16]."""
    nb, hkv, d = _q8_pool_dims(k_codes, v_codes, k_scales, v_scales)
    dev = k_codes.device
    _need(k, "k", torch.bfloat16, 3, dev)
    _need(v, "v", torch.bfloat16, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    T = slot_mapping.shape[0]
    if k.shape != (T, hkv, d) or v.shape != k.shape:
        raise ValueError("k/v must be [num_tokens, num_kv_heads, head_dim]")
    dims = _dims(0, 0, hkv, d, nb, 0)
    check("pkv_kv_append_q8", load().pkv_kv_append_q8(
        _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), _ptr(k), _ptr(v), _ptr(slot_mapping), T,
        ctypes.byref(dims), _ptr(error_word), _stream(stream, dev)))


def decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, num_blocks,
                           max_blocks_per_seq) -> int:
    dims = _dims(batch, num_q_heads, num_kv_heads, head_dim, num_blocks, max_blocks_per_seq)
    n = load().pkv_decode_workspace_bytes(ctypes.byref(dims))
    if n == 0:
        raise ValueError("invalid dims for paged decode")
    return int(n)


def sparse_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, num_blocks,
                                  max_blocks_per_seq, max_kept) -> int:
    dims = _dims(batch, num_q_heads, num_kv_heads, head_dim, num_blocks, max_blocks_per_seq)
    n = load().pkv_sparse_decode_workspace_bytes(ctypes.byref(dims), int(max_kept))
    if n == 0:
        raise ValueError("invalid dims for sparse decode")
    return int(n)


def _flags(inputs_ready: bool) -> int:
    """The decode calls' flags word: PKV_DECODE_INPUTS_READY when the caller declares the pools,
    block tables, lengths (and kept lists) final before the preceding work on the stream."""
    return _INPUTS_READY if inputs_ready else 0


def _decode_inputs(q, k_cache, v_cache, block_tables, context_lens):
    nb, hkv, d = _pool_dims(k_cache, v_cache)
    dev = k_cache.device
    _need(q, "q", torch.bfloat16, 3, dev, host_ok=True)
    _need(block_tables, "block_tables", torch.int32, 2, dev, host_ok=True)
    _need(context_lens, "context_lens", torch.int32, 1, dev, host_ok=True)
    B, hq, dq = q.shape
    if dq != d:
        raise ValueError("q head_dim differs from the pools'")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens batch differs from q's")
    return _dims(B, hq, hkv, d, nb, block_tables.shape[1]), dev


def _out_ws(q, out, workspace, nbytes, dev):
    """out (given: on dev or in pinned host memory; else allocated on dev) and the workspace."""
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=dev)
    else:
        _need(out, "out", torch.bfloat16, 3, dev, host_ok=True)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if workspace is None:
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    else:
        _need(workspace, "workspace", torch.uint8, 1, dev)
    return out, workspace


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale, window=0, *,
                           out=None, workspace=None, error_word=None, inputs_ready=False, stream=None):
    """softmax(scale * q K^T) V over the paged cache; returns out [B, Hq, d] bf16."""
    dims, dev = _decode_inputs(q, k_cache, v_cache, block_tables, context_lens)
    nbytes = int(load().pkv_decode_workspace_bytes(ctypes.byref(dims)))
    out, workspace = _out_ws(q, out, workspace, nbytes, dev)
    check("pkv_paged_decode_attention", load().pkv_paged_decode_attention(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        float(scale), int(window), _ptr(workspace), workspace.numel(), ctypes.byref(dims),
        _flags(inputs_ready), _ptr(error_word), _stream(stream, dev)))
    return out


def _q8_decode_inputs(q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens):
    nb, hkv, d = _q8_pool_dims(k_codes, v_codes, k_scales, v_scales)
    dev = k_codes.device
    _need(q, "q", torch.bfloat16, 3, dev, host_ok=True)
    _need(block_tables, "block_tables", torch.int32, 2, dev, host_ok=True)
    _need(context_lens, "context_lens", torch.int32, 1, dev, host_ok=True)
    B, hq, dq = q.shape
    if dq != d:
        raise ValueError("q head_dim differs from the pools'")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens batch differs from q's")
    return _dims(B, hq, hkv, d, nb, block_tables.shape[1]), dev


def paged_decode_attention_q8(q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens, scale,
                              window=0, *, out=None, workspace=None, error_word=None, inputs_ready=False, stream=None):
    """paged_decode_attention over INT8 pools (each element code * its row's scale)."""
    dims, dev = _q8_decode_inputs(q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens)
    nbytes = int(load().pkv_decode_workspace_bytes(ctypes.byref(dims)))
    out, workspace = _out_ws(q, out, workspace, nbytes, dev)
    check("pkv_paged_decode_attention_q8", load().pkv_paged_decode_attention_q8(
        _ptr(out), _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), _ptr(block_tables),
        _ptr(context_lens), float(scale), int(window), _ptr(workspace), workspace.numel(), ctypes.byref(dims),
        _flags(inputs_ready), _ptr(error_word), _stream(stream, dev)))
    return out


def prefill_window_scores(q_win, k_cache, block_tables, context_lens, scale, score_accum, *, lse=None,
                          lse_given=False, error_word=None, stream=None):
    """Add the prefill-window score of every prompt key into score_accum [B, Hkv, S] (fp32).
    q_win [B, alpha, Hq, d] bf16 holds the queries of the last alpha prompt positions.  lse
    [B, Hq, alpha] fp32: read when lse_given (the prefill attention's log-sum-exps), else
    computed into it (allocated when None).  Returns lse."""
    nb, hkv, d = _pool_dims(k_cache, k_cache)
    dev = k_cache.device
    _need(q_win, "q_win", torch.bfloat16, 4, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    _need(score_accum, "score_accum", torch.float32, 3, dev)
    B, alpha, hq, dq = q_win.shape
    if dq != d:
        raise ValueError("q_win head_dim differs from the pool's")
    if block_tables.shape[0] != B or context_lens.shape[0] != B or score_accum.shape[:2] != (B, hkv):
        raise ValueError("batch / kv heads of block_tables, context_lens or score_accum differ from q_win's")
    if lse is None:
        if lse_given:
            raise ValueError("lse_given needs lse")
        lse = torch.empty((B, hq, alpha), dtype=torch.float32, device=dev)
    else:
        _need(lse, "lse", torch.float32, 3, dev)
        if lse.shape != (B, hq, alpha):
            raise ValueError("lse must be [B, Hq, alpha]")
    dims = _dims(B, hq, hkv, d, nb, block_tables.shape[1])
    check("pkv_prefill_window_scores", load().pkv_prefill_window_scores(
        _ptr(score_accum), score_accum.shape[2], _ptr(lse), int(bool(lse_given)), _ptr(q_win), _ptr(k_cache),
        _ptr(block_tables), _ptr(context_lens), int(alpha), float(scale), ctypes.byref(dims), _ptr(error_word),
        _stream(stream, dev)))
    return lse


def paged_decode_attention_append(q, k_cache, v_cache, k_new, v_new, block_tables, context_lens,
                                  scale, window=0, *, out=None, workspace=None, error_word=None, inputs_ready=False,
                                  stream=None):
    """One decode step: write k_new/v_new [B, Hkv, d] at each sequence's last position
    (context_lens[b] - 1, through the block table) and attend, in one kernel.  Same result as
    kv_append followed by paged_decode_attention for that slot layout."""
    dims, dev = _decode_inputs(q, k_cache, v_cache, block_tables, context_lens)
    _need(k_new, "k_new", torch.bfloat16, 3, dev, host_ok=True)
    _need(v_new, "v_new", torch.bfloat16, 3, dev, host_ok=True)
    if k_new.shape != (dims.batch, dims.num_kv_heads, dims.head_dim) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [B, Hkv, head_dim]")
    nbytes = int(load().pkv_decode_workspace_bytes(ctypes.byref(dims)))
    out, workspace = _out_ws(q, out, workspace, nbytes, dev)
    check("pkv_paged_decode_attention_append", load().pkv_paged_decode_attention_append(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
        _ptr(block_tables), _ptr(context_lens), float(scale), int(window), _ptr(workspace),
        workspace.numel(), ctypes.byref(dims), _flags(inputs_ready), _ptr(error_word), _stream(stream, dev)))
    return out


def _score_buffers(dims, dev, score_accum, lse, logits):
    """Checks score_accum [B, Hkv, S]; returns (S, lse [B, Hq], logits [B, Hq, S]), allocating
    the last two when not given."""
    _need(score_accum, "score_accum", torch.float32, 3, dev)
    if score_accum.shape[:2] != (dims.batch, dims.num_kv_heads):
        raise ValueError("score_accum must be [B, Hkv, S]")
    stride = score_accum.shape[2]
    if lse is None:
        lse = torch.empty((dims.batch, dims.num_q_heads), dtype=torch.float32, device=dev)
    else:
        _need(lse, "lse", torch.float32, 2, dev)
        if lse.shape != (dims.batch, dims.num_q_heads):
            raise ValueError("lse must be [B, Hq]")
    if logits is None:
        logits = torch.empty((dims.batch, dims.num_q_heads, stride), dtype=torch.float32, device=dev)
    else:
        _need(logits, "logits", torch.float32, 3, dev)
        if logits.shape != (dims.batch, dims.num_q_heads, stride):
            raise ValueError("logits must be [B, Hq, S]")
    return stride, lse, logits


def paged_decode_attention_scores(q, k_cache, v_cache, block_tables, context_lens, scale, score_accum,
                                  window=0, *, k_new=None, v_new=None, out=None, lse=None, logits=None,
                                  workspace=None, error_word=None, inputs_ready=False, stream=None):
    """paged_decode_attention (with the step's append when k_new/v_new are given) that also
    adds the step's sparsification score into score_accum [B, Hkv, S] fp32: for every attended
    key t < S of (b, kv head g), the sum over g's query heads of their softmax probability of
    t.  Returns (out [B, Hq, d] bf16, lse [B, Hq] fp32: each row's natural log-sum-exp).
    logits [B, Hq, S] fp32 is scratch (allocated when not given)."""
    dims, dev = _decode_inputs(q, k_cache, v_cache, block_tables, context_lens)
    stride, lse, logits = _score_buffers(dims, dev, score_accum, lse, logits)
    if (k_new is None) != (v_new is None):
        raise ValueError("give both k_new and v_new, or neither")
    if k_new is not None:
        _need(k_new, "k_new", torch.bfloat16, 3, dev, host_ok=True)
        _need(v_new, "v_new", torch.bfloat16, 3, dev, host_ok=True)
        if k_new.shape != (dims.batch, dims.num_kv_heads, dims.head_dim) or v_new.shape != k_new.shape:
            raise ValueError("k_new/v_new must be [B, Hkv, head_dim]")
    nbytes = int(load().pkv_decode_workspace_bytes(ctypes.byref(dims)))
    out, workspace = _out_ws(q, out, workspace, nbytes, dev)
    check("pkv_paged_decode_attention_scores", load().pkv_paged_decode_attention_scores(
        _ptr(out), _ptr(lse), _ptr(score_accum), _ptr(logits), int(stride), _ptr(q), _ptr(k_cache),
        _ptr(v_cache), _ptr(k_new), _ptr(v_new), _ptr(block_tables), _ptr(context_lens), float(scale),
        int(window), _ptr(workspace), workspace.numel(), ctypes.byref(dims), _flags(inputs_ready), _ptr(error_word),
        _stream(stream, dev)))
    return out, lse


def paged_decode_attention_append_q8(q, k_codes, v_codes, k_scales, v_scales, k_new, v_new, block_tables,
                                     context_lens, scale, window=0, *, out=None, workspace=None, error_word=None, inputs_ready=False,
                                     stream=None):
    """kv_append_q8 of k_new/v_new [B, Hkv, d] (bf16) at each sequence's position L_b - 1, fused
    into paged_decode_attention_q8 over the updated INT8 pools."""
    dims, dev = _q8_decode_inputs(q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens)
    _need(k_new, "k_new", torch.bfloat16, 3, dev, host_ok=True)
    _need(v_new, "v_new", torch.bfloat16, 3, dev, host_ok=True)
    if k_new.shape != (dims.batch, dims.num_kv_heads, dims.head_dim) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [B, Hkv, head_dim]")
    nbytes = int(load().pkv_decode_workspace_bytes(ctypes.byref(dims)))
    out, workspace = _out_ws(q, out, workspace, nbytes, dev)
    check("pkv_paged_decode_attention_append_q8", load().pkv_paged_decode_attention_append_q8(
        _ptr(out), _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), _ptr(k_new), _ptr(v_new),
        _ptr(block_tables), _ptr(context_lens), float(scale), int(window), _ptr(workspace), workspace.numel(),
        ctypes.byref(dims), _flags(inputs_ready), _ptr(error_word), _stream(stream, dev)))
    return out


def sparse_decode_attention_q8(q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens,
                               kept_index_lists, kept_lens, scale, *, out=None, workspace=None, error_word=None, inputs_ready=False,
                               stream=None):
    """sparse_decode_attention over INT8 pools (each element code * its row's scale)."""
    dims, dev = _q8_decode_inputs(q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens)
    _need(kept_index_lists, "kept_index_lists", torch.int32, 3, dev)
    _need(kept_lens, "kept_lens", torch.int32, 1, dev)
    if kept_index_lists.shape[:2] != (dims.batch, dims.num_kv_heads) or kept_lens.shape[0] != dims.batch:
        raise ValueError("kept_index_lists must be [B, Hkv, max_kept] and kept_lens [B]")
    max_kept = kept_index_lists.shape[2]
    nbytes = int(load().pkv_sparse_decode_workspace_bytes(ctypes.byref(dims), max_kept))
    out, workspace = _out_ws(q, out, workspace, nbytes, dev)
    check("pkv_sparse_decode_attention_q8", load().pkv_sparse_decode_attention_q8(
        _ptr(out), _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), _ptr(block_tables),
        _ptr(context_lens), _ptr(kept_index_lists), _ptr(kept_lens), max_kept, float(scale), _ptr(workspace),
        workspace.numel(), ctypes.byref(dims), _flags(inputs_ready), _ptr(error_word), _stream(stream, dev)))
    return out


def paged_decode_attention_scores_q8(q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens, scale,
                                     score_accum, window=0, *, out=None, lse=None, logits=None, workspace=None,
                                     error_word=None, inputs_ready=False, stream=None):
    """paged_decode_attention_scores over INT8 pools (no append: INT8 pools take the step's
    token through kv_append_q8).  Returns (out, lse) as paged_decode_attention_scores."""
    dims, dev = _q8_decode_inputs(q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens)
    stride, lse, logits = _score_buffers(dims, dev, score_accum, lse, logits)
    nbytes = int(load().pkv_decode_workspace_bytes(ctypes.byref(dims)))
    out, workspace = _out_ws(q, out, workspace, nbytes, dev)
    check("pkv_paged_decode_attention_scores_q8", load().pkv_paged_decode_attention_scores_q8(
        _ptr(out), _ptr(lse), _ptr(score_accum), _ptr(logits), int(stride), _ptr(q), _ptr(k_codes), _ptr(v_codes),
        _ptr(k_scales), _ptr(v_scales), _ptr(block_tables), _ptr(context_lens), float(scale), int(window),
        _ptr(workspace), workspace.numel(), ctypes.byref(dims), _flags(inputs_ready), _ptr(error_word), _stream(stream, dev)))
    return out, lse


def kv_rolling_admit(k_cache, v_cache, block_tables, slot_pos, slot_score, kept_lens, context_lens, k_new,
                     v_new, n_sink, n_recent, *, error_word=None, inputs_ready=False, stream=None):
    """Admit this step's token (k_new/v_new [B, Hkv, d], position context_lens[b] - 1) into each
    sequence's fixed-budget sparse cache: the compact pool [NB, Hkv, 16, d] with its tables,
    slot_pos [B, Hkv, C] int32 and slot_score [B, Hkv, C] fp32 (C = n_sink + k_top + n_recent
    slots) and kept_lens [B] int32, all updated in place.  See pkv_kv_rolling_admit.
    inputs_ready=True sets PKV_ADMIT_INPUTS_READY: the slot state, lengths and tables are final
    before the preceding work on the stream, so the slots are chosen before that work ends."""
    nb, hkv, d = _pool_dims(k_cache, v_cache)
    dims = _rolling_dims(nb, hkv, d, k_cache.device, block_tables, slot_pos, slot_score, kept_lens, context_lens,
                         k_new, v_new)
    check("pkv_kv_rolling_admit", load().pkv_kv_rolling_admit(
        _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(slot_pos), _ptr(slot_score), _ptr(kept_lens),
        _ptr(context_lens), _ptr(k_new), _ptr(v_new), slot_pos.shape[2], int(n_sink), int(n_recent),
        ctypes.byref(dims), _ADMIT_READY if inputs_ready else 0, _ptr(error_word), _stream(stream, k_cache.device)))


def kv_rolling_admit_q8(k_codes, v_codes, k_scales, v_scales, block_tables, slot_pos, slot_score, kept_lens,
                        context_lens, k_new, v_new, n_sink, n_recent, *, error_word=None, inputs_ready=False,
                        stream=None):
    """kv_rolling_admit into INT8 compact pools (codes [NB, Hkv, 16, d] uint8 as code + 128, row scales
    [NB, Hkv, 16] fp32): the same slot choice, the new rows quantized into the slot (inputs_ready as
    kv_rolling_admit)."""
    nb, hkv, d = _q8_pool_dims(k_codes, v_codes, k_scales, v_scales)
    dims = _rolling_dims(nb, hkv, d, k_codes.device, block_tables, slot_pos, slot_score, kept_lens, context_lens,
                         k_new, v_new)
    check("pkv_kv_rolling_admit_q8", load().pkv_kv_rolling_admit_q8(
        _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), _ptr(block_tables), _ptr(slot_pos),
        _ptr(slot_score), _ptr(kept_lens), _ptr(context_lens), _ptr(k_new), _ptr(v_new), slot_pos.shape[2],
        int(n_sink), int(n_recent), ctypes.byref(dims), _ADMIT_READY if inputs_ready else 0, _ptr(error_word),
        _stream(stream, k_codes.device)))


def _rolling_dims(nb, hkv, d, dev, block_tables, slot_pos, slot_score, kept_lens, context_lens, k_new, v_new):
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(slot_pos, "slot_pos", torch.int32, 3, dev)
    _need(slot_score, "slot_score", torch.float32, 3, dev)
    _need(kept_lens, "kept_lens", torch.int32, 1, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    _need(k_new, "k_new", torch.bfloat16, 3, dev, host_ok=True)
    _need(v_new, "v_new", torch.bfloat16, 3, dev, host_ok=True)
    B = slot_pos.shape[0]
    if slot_pos.shape[1] != hkv or slot_score.shape != slot_pos.shape:
        raise ValueError("slot_pos and slot_score must be [B, Hkv, capacity]")
    if k_new.shape != (B, hkv, d) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [B, Hkv, head_dim]")
    if block_tables.shape[0] != B or kept_lens.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / kept_lens / context_lens batch differs")
    return _dims(B, 1, hkv, d, nb, block_tables.shape[1])


def paged_decode_attention_fixed_scratch(q, k_cache, v_cache, block_tables, context_lens, scale,
                                         window=0, *, out=None, error_word=None, stream=None):
    """paged_decode_attention without a workspace, for callers that cannot allocate device
    memory: the library's fixed static scratch (PKV_FIXED_SCRATCH_BYTES) holds the split-K
    partials.  Shapes that need more scratch are refused.  Calls that overlap on the GPU
    share that scratch and race; issue them one after another.  (Only `out`, when not
    given, is allocated here by torch; pass it to allocate nothing.)"""
    dims, dev = _decode_inputs(q, k_cache, v_cache, block_tables, context_lens)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=dev)
    else:
        _need(out, "out", torch.bfloat16, 3, dev, host_ok=True)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    check("pkv_paged_decode_attention_fixed_scratch",
          load().pkv_paged_decode_attention_fixed_scratch(
              _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
              _ptr(context_lens), float(scale), int(window), ctypes.byref(dims), _ptr(error_word),
              _stream(stream, dev)))
    return out


def sparse_decode_attention(q, k_cache, v_cache, block_tables, context_lens, kept_index_lists,
                            kept_lens, scale, *, out=None, workspace=None, error_word=None, inputs_ready=False,
                            stream=None):
    """Decode attention over kept_index_lists [B, Hkv, max_kept][:kept_lens[b]]."""
    dims, dev = _decode_inputs(q, k_cache, v_cache, block_tables, context_lens)
    _need(kept_index_lists, "kept_index_lists", torch.int32, 3, dev)
    _need(kept_lens, "kept_lens", torch.int32, 1, dev)
    if kept_index_lists.shape[:2] != (dims.batch, dims.num_kv_heads):
        raise ValueError("kept_index_lists must be [B, Hkv, max_kept]")
    max_kept = kept_index_lists.shape[2]
    nbytes = int(load().pkv_sparse_decode_workspace_bytes(ctypes.byref(dims), max_kept))
    out, workspace = _out_ws(q, out, workspace, nbytes, dev)
    check("pkv_sparse_decode_attention", load().pkv_sparse_decode_attention(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        _ptr(kept_index_lists), _ptr(kept_lens), max_kept, float(scale), _ptr(workspace),
        workspace.numel(), ctypes.byref(dims), _flags(inputs_ready), _ptr(error_word), _stream(stream, dev)))
    return out


def kv_select_topk(score_accum, context_lens, n_sink, n_recent, k_top, *, kept_out=None,
                   kept_lens_out=None, error_word=None, inputs_ready=False, stream=None):
    """Kept positions per (sequence, kv head): sinks, top-k by score, recent window.

    score_accum [B, Hkv, S] fp32 -> (kept [B, Hkv, n_sink+k_top+n_recent] int32 ascending,
    kept_lens [B] int32); entries past kept_lens[b] are left as they were (-1 when allocated here).
    inputs_ready: PKV_SELECT_INPUTS_READY (the scores and lengths are final before the work
    enqueued just before this call ends; results are identical).
    """
    _need(score_accum, "score_accum", torch.float32, 3)
    dev = score_accum.device
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    B, hkv, stride = score_accum.shape
    kmax = int(n_sink) + int(k_top) + int(n_recent)
    if kept_out is None:
        kept_out = torch.full((B, hkv, kmax), -1, dtype=torch.int32, device=dev)
    else:
        _need(kept_out, "kept_out", torch.int32, 3, dev)
        if kept_out.shape != (B, hkv, kmax):
            raise ValueError("kept_out must be [B, Hkv, n_sink + k_top + n_recent]")
    if kept_lens_out is None:
        kept_lens_out = torch.empty(B, dtype=torch.int32, device=dev)
    else:
        _need(kept_lens_out, "kept_lens_out", torch.int32, 1, dev)
    dims = _dims(B, hkv, hkv, 128, 0, 0)
    check("pkv_kv_select_topk", load().pkv_kv_select_topk(
        _ptr(kept_out), _ptr(kept_lens_out), _ptr(score_accum), stride, _ptr(context_lens),
        int(n_sink), int(n_recent), int(k_top), ctypes.byref(dims), _SELECT_READY if inputs_ready else 0,
        _ptr(error_word), _stream(stream, dev)))
    return kept_out, kept_lens_out


def kv_compact(dst_k_cache, dst_v_cache, dst_block_tables, src_k_cache, src_v_cache,
               src_block_tables, context_lens, kept_index_lists, kept_lens, *, error_word=None,
               inputs_ready=False, stream=None):
    """Copy each (sequence, kv head)'s kept tokens into consecutive slots of the dst pool.

    inputs_ready=True sets PKV_COMPACT_INPUTS_READY: the caller declares the source pools and
    tables, the lengths, the kept lists and dst_block_tables final before the preceding work on
    the stream (not written by it), so the call reads the kept rows before that work ends."""
    snb, hkv, d = _pool_dims(src_k_cache, src_v_cache)
    dnb, dhkv, dd = _pool_dims(dst_k_cache, dst_v_cache)
    if (dhkv, dd) != (hkv, d):
        raise ValueError("source and destination pools differ in heads or head_dim")
    dev = src_k_cache.device
    _need(dst_block_tables, "dst_block_tables", torch.int32, 2, dev)
    _need(src_block_tables, "src_block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    _need(kept_index_lists, "kept_index_lists", torch.int32, 3, dev)
    _need(kept_lens, "kept_lens", torch.int32, 1, dev)
    B = kept_index_lists.shape[0]
    if kept_index_lists.shape[1] != hkv:
        raise ValueError("kept_index_lists must be [B, Hkv, max_kept]")
    dims = _dims(B, hkv, hkv, d, snb, src_block_tables.shape[1])
    check("pkv_kv_compact", load().pkv_kv_compact(
        _ptr(dst_k_cache), _ptr(dst_v_cache), _ptr(dst_block_tables), dnb, dst_block_tables.shape[1],
        _ptr(src_k_cache), _ptr(src_v_cache), _ptr(src_block_tables), _ptr(context_lens),
        _ptr(kept_index_lists), _ptr(kept_lens), kept_index_lists.shape[2], ctypes.byref(dims),
        _COMPACT_READY if inputs_ready else 0, _ptr(error_word), _stream(stream, dev)))


def kv_compact_q8(dst_k_codes, dst_v_codes, dst_k_scales, dst_v_scales, dst_block_tables, src_k_codes,
                  src_v_codes, src_k_scales, src_v_scales, src_block_tables, context_lens, kept_index_lists,
                  kept_lens, *, error_word=None, inputs_ready=False, stream=None):
    """kv_compact over INT8 pools: each kept row's codes and row scale move together
    (inputs_ready as kv_compact)."""
    snb, hkv, d = _q8_pool_dims(src_k_codes, src_v_codes, src_k_scales, src_v_scales)
    dnb, dhkv, dd = _q8_pool_dims(dst_k_codes, dst_v_codes, dst_k_scales, dst_v_scales)
    if (dhkv, dd) != (hkv, d):
        raise ValueError("source and destination pools differ in heads or head_dim")
    dev = src_k_codes.device
    if dst_k_codes.device != dev:
        raise ValueError("source and destination pools are on different devices")
    _need(dst_block_tables, "dst_block_tables", torch.int32, 2, dev)
    _need(src_block_tables, "src_block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    _need(kept_index_lists, "kept_index_lists", torch.int32, 3, dev)
    _need(kept_lens, "kept_lens", torch.int32, 1, dev)
    B = kept_index_lists.shape[0]
    if kept_index_lists.shape[1] != hkv:
        raise ValueError("kept_index_lists must be [B, Hkv, max_kept]")
    dims = _dims(B, hkv, hkv, d, snb, src_block_tables.shape[1])
    check("pkv_kv_compact_q8", load().pkv_kv_compact_q8(
        _ptr(dst_k_codes), _ptr(dst_v_codes), _ptr(dst_k_scales), _ptr(dst_v_scales), _ptr(dst_block_tables), dnb,
        dst_block_tables.shape[1], _ptr(src_k_codes), _ptr(src_v_codes), _ptr(src_k_scales), _ptr(src_v_scales),
        _ptr(src_block_tables), _ptr(context_lens), _ptr(kept_index_lists), _ptr(kept_lens),
        kept_index_lists.shape[2], ctypes.byref(dims), _COMPACT_READY if inputs_ready else 0, _ptr(error_word),
        _stream(stream, dev)))
