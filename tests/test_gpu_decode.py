"""GPU parity of kv_append and paged_decode_attention (through the C ABI) against the fp64
oracle.  Small cases compare every output element; the full-size workloads run in the launch
configuration the bench times and compare a deterministic sample of rows the oracle computes
one by one.  Tolerance: max-abs 1e-2 and relative L2 2e-3 (bf16 in, fp32 accumulate, bf16 out);
append is bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_mapped_gb300 as pkv
from paged_kv_cache_mapped_gb300 import inputs as W
from helpers import assert_attn_close, bits, paged_from_contiguous, rand_bf16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _oracle_rows(case, rows, kc_bits=None, vc_bits=None, window=0):
    return oracle.paged_decode(bits(case["q"]), bits(case["k_cache"]) if kc_bits is None else kc_bits,
                               bits(case["v_cache"]) if vc_bits is None else vc_bits,
                               case["block_tables"].cpu().numpy(), case["context_lens"].cpu().numpy(),
                               case["scale"], window, rows=rows)


def _run(case, window=0, err=None):
    out = pkv.paged_decode_attention(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                                     case["context_lens"], case["scale"], window, error_word=err)
    torch.cuda.synchronize()
    return out


def _small_case(lens, hq, hkv, d, seed, fill=None, nb_extra=5):
    g = torch.Generator().manual_seed(seed)
    B = len(lens)
    lmax = max(max(lens), 1)
    k = rand_bf16((B, lmax, hkv, d), g)
    v = rand_bf16((B, lmax, hkv, d), g)
    q = rand_bf16((B, hq, d), g)
    nb = sum((L + 15) // 16 for L in lens) + nb_extra
    kc, vc, bt = paged_from_contiguous(k, v, lens, nb, g, fill=fill)
    return {"q": q.to(DEV), "k_cache": kc.to(DEV), "v_cache": vc.to(DEV), "block_tables": bt.to(DEV),
            "context_lens": torch.tensor(lens, dtype=torch.int32, device=DEV), "scale": d ** -0.5}


@pytest.mark.parametrize("window", [0, 1, 16, 50, 100, 300])
def test_tiny_workload_every_element(window):
    wl = W.WORKLOADS["tiny"]
    case = W.make_layer(wl, device=DEV)
    err = pkv.new_error_word(DEV)
    out = _run(case, window, err)
    assert pkv.read_error(err) == 0
    ref = _oracle_rows(case, None, window=window)
    assert_attn_close(out, ref, f"tiny window={window}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 6, 8])
def test_ragged_lengths_all_groups(d, group):
    hkv = 2
    lens = [1, 15, 16, 17, 33, 100, 257, 1000, 2049]
    case = _small_case(lens, hq=hkv * group, hkv=hkv, d=d, seed=d + group)
    for window in (0, 7, 40):
        out = _run(case, window)
        assert_attn_close(out, _oracle_rows(case, None, window=window), f"d={d} G={group} w={window}")


def test_unused_slots_hold_nan():
    case = _small_case([5, 17, 31, 64, 200], hq=8, hkv=2, d=128, seed=3, fill=float("nan"))
    for window in (0, 9):
        out = _run(case, window)
        assert_attn_close(out, _oracle_rows(case, None, window=window), f"nan poison w={window}")


def test_empty_sequences_give_zero_rows():
    case = _small_case([0, 40, 0, 3], hq=4, hkv=2, d=64, seed=4)
    out = _run(case)
    assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[2]) == 0
    ref = _oracle_rows(case, None)
    assert_attn_close(out, ref, "empty rows")


def test_single_token_exact_and_equal_rows():
    # one attended token: the output is that token's V row exactly (bf16 -> fp32 -> bf16)
    case = _small_case([1, 1, 1], hq=8, hkv=2, d=128, seed=5)
    out = _run(case)
    bt = case["block_tables"].cpu()
    for b in range(3):
        blk = int(bt[b, 0])
        for h in range(8):
            assert torch.equal(out[b, h].cpu(), case["v_cache"][blk, h // 4, 0].cpu())
    # window 1 over long contexts: the last token's V exactly
    case = _small_case([300, 513], hq=4, hkv=4, d=64, seed=6)
    out = _run(case, window=1)
    bt = case["block_tables"].cpu()
    for b, L in enumerate([300, 513]):
        blk = int(bt[b, (L - 1) // 16])
        for h in range(4):
            assert torch.equal(out[b, h].cpu(), case["v_cache"][blk, h, (L - 1) % 16].cpu())


def test_deterministic_and_workspace_reuse():
    case = _small_case([700, 33, 1500], hq=8, hkv=2, d=128, seed=7)
    ws = torch.zeros(pkv.decode_workspace_bytes(3, 8, 2, 128, case["k_cache"].shape[0],
                                                case["block_tables"].shape[1]),
                     dtype=torch.uint8, device=DEV)
    a = pkv.paged_decode_attention(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                                   case["context_lens"], case["scale"], workspace=ws)
    b = pkv.paged_decode_attention(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                                   case["context_lens"], case["scale"], workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_bad_block_id_sets_error_word():
    case = _small_case([100, 60], hq=4, hkv=2, d=128, seed=8)
    case["block_tables"][1, 2] = case["k_cache"].shape[0] + 5
    err = pkv.new_error_word(DEV)
    out = _run(case, err=err)
    assert pkv.read_error(err, clear=True) == pkv.header_constants()["PKV_DEV_BAD_BLOCK_ID"]
    assert torch.isfinite(out.float()).all()
    # the untouched sequence is still right
    ref = _oracle_rows(case, list(range(0, 4)))
    assert_attn_close(out[0], ref, "valid sequence next to a bad one")
    assert pkv.read_error(err) == 0


def test_bad_context_len_sets_error_word():
    case = _small_case([100, 60], hq=4, hkv=2, d=64, seed=9)
    case["context_lens"][1] = case["block_tables"].shape[1] * 16 + 1
    err = pkv.new_error_word(DEV)
    out = _run(case, err=err)
    assert pkv.read_error(err) == pkv.header_constants()["PKV_DEV_BAD_CONTEXT_LEN"]
    assert torch.count_nonzero(out[1]) == 0


def _sample_rows(B, hq, n, seed):
    rng = np.random.default_rng(seed)
    rows = {0, B * hq - 1}
    rows |= {b * hq for b in range(B)}
    rows |= set(rng.choice(B * hq, size=min(n, B * hq), replace=False).tolist())
    return sorted(rows)


def test_llama8b_full_size_append_then_decode():
    wl = W.WORKLOADS["llama8b"]
    case = W.make_layer(wl, device=DEV)
    kc0, vc0 = bits(case["k_cache"]), bits(case["v_cache"])
    err = pkv.new_error_word(DEV)
    pkv.kv_append(case["k_cache"], case["v_cache"], case["k_new"], case["v_new"], case["slot_mapping"],
                  error_word=err)
    out = _run(case, err=err)
    assert pkv.read_error(err) == 0
    okc, ovc = oracle.kv_append(kc0, vc0, bits(case["k_new"]), bits(case["v_new"]),
                                case["slot_mapping"].cpu().numpy())
    assert np.array_equal(bits(case["k_cache"]), okc)
    assert np.array_equal(bits(case["v_cache"]), ovc)
    rows = _sample_rows(wl.batch, wl.num_q_heads, 64, 2)
    ref = _oracle_rows(case, rows, okc, ovc)
    got = out.view(-1, wl.head_dim)[torch.tensor(rows, device=DEV)]
    assert_attn_close(got, ref, "llama8b sampled rows")


@pytest.mark.parametrize("layer", [0, 27])
def test_qwen_layers_full_size(layer):
    wl = W.WORKLOADS["qwen1p5b"]
    case = W.make_layer(wl, layer=layer, device=DEV)
    kc0, vc0 = bits(case["k_cache"]), bits(case["v_cache"])
    pkv.kv_append(case["k_cache"], case["v_cache"], case["k_new"], case["v_new"], case["slot_mapping"])
    out = _run(case)
    okc, ovc = oracle.kv_append(kc0, vc0, bits(case["k_new"]), bits(case["v_new"]),
                                case["slot_mapping"].cpu().numpy())
    assert np.array_equal(bits(case["k_cache"]), okc)
    rows = _sample_rows(wl.batch, wl.num_q_heads, 96, 3 + layer)
    ref = _oracle_rows(case, rows, okc, ovc)
    got = out.view(-1, wl.head_dim)[torch.tensor(rows, device=DEV)]
    assert_attn_close(got, ref, f"qwen layer {layer}")


def test_long128k_full_size_sampled():
    wl = W.WORKLOADS["long128k"]
    case = W.make_layer(wl, device=DEV, device_rng=True)
    err = pkv.new_error_word(DEV)
    out = _run(case, err=err)
    assert pkv.read_error(err) == 0
    rows = _sample_rows(wl.batch, wl.num_q_heads, 12, 4)
    ref = _oracle_rows(case, rows)
    got = out.view(-1, wl.head_dim)[torch.tensor(rows, device=DEV)]
    assert_attn_close(got, ref, "long128k sampled rows")
    # a sliding window over the same long context
    out_w = _run(case, window=4096)
    ref_w = _oracle_rows(case, rows, window=4096)
    assert_attn_close(out_w.view(-1, wl.head_dim)[torch.tensor(rows, device=DEV)], ref_w, "long128k w=4096")


@pytest.mark.parametrize("window", [0, 5])
def test_fused_append_decode_small_ragged(window):
    """paged_decode_attention_append == kv_append at position L-1 then paged decode (oracle)."""
    lens = [1, 15, 16, 17, 33, 100, 257]
    for d, hq, hkv in ((128, 8, 2), (64, 6, 3)):
        case = _small_case(lens, hq=hq, hkv=hkv, d=d, seed=31 + d, fill=float("nan"))
        g = torch.Generator().manual_seed(32)
        k_new = rand_bf16((len(lens), hkv, d), g)
        v_new = rand_bf16((len(lens), hkv, d), g)
        bt = case["block_tables"].cpu()
        slots = np.array([int(bt[b, (L - 1) // 16]) * 16 + (L - 1) % 16 for b, L in enumerate(lens)],
                         dtype=np.int64)
        okc, ovc = oracle.kv_append(bits(case["k_cache"]), bits(case["v_cache"]), bits(k_new), bits(v_new),
                                    slots)
        err = pkv.new_error_word(DEV)
        out = pkv.paged_decode_attention_append(case["q"], case["k_cache"], case["v_cache"], k_new.to(DEV),
                                                v_new.to(DEV), case["block_tables"], case["context_lens"],
                                                case["scale"], window, error_word=err)
        torch.cuda.synchronize()
        assert pkv.read_error(err) == 0
        assert np.array_equal(bits(case["k_cache"]), okc) and np.array_equal(bits(case["v_cache"]), ovc)
        ref = _oracle_rows(case, None, okc, ovc, window=window)
        assert_attn_close(out, ref, f"fused append d={d} w={window}")


def test_fused_append_decode_llama8b_full_size():
    wl = W.WORKLOADS["llama8b"]
    case = W.make_layer(wl, device=DEV, device_rng=True)
    kc0, vc0 = bits(case["k_cache"]), bits(case["v_cache"])
    err = pkv.new_error_word(DEV)
    out = pkv.paged_decode_attention_append(case["q"], case["k_cache"], case["v_cache"], case["k_new"],
                                            case["v_new"], case["block_tables"], case["context_lens"],
                                            case["scale"], error_word=err)
    torch.cuda.synchronize()
    assert pkv.read_error(err) == 0
    okc, ovc = oracle.kv_append(kc0, vc0, bits(case["k_new"]), bits(case["v_new"]),
                                case["slot_mapping"].cpu().numpy())
    assert np.array_equal(bits(case["k_cache"]), okc) and np.array_equal(bits(case["v_cache"]), ovc)
    rows = _sample_rows(wl.batch, wl.num_q_heads, 64, 12)
    ref = _oracle_rows(case, rows, okc, ovc)
    got = out.view(-1, wl.head_dim)[torch.tensor(rows, device=DEV)]
    assert_attn_close(got, ref, "llama8b fused append sampled rows")


def test_workspace_reused_across_shapes():
    """One zero-filled workspace serves calls of different batch sizes and head counts in turn
    (every call leaves the ticket counters at its start zero)."""
    cases = [_small_case([700, 33, 1500], hq=8, hkv=2, d=128, seed=41),
             _small_case([90] * 16, hq=16, hkv=4, d=128, seed=42),
             _small_case([5000, 1, 2500, 17], hq=32, hkv=8, d=128, seed=43),
             _small_case([700, 33, 1500], hq=8, hkv=2, d=128, seed=41)]
    need = max(pkv.decode_workspace_bytes(c["q"].shape[0], c["q"].shape[1], c["k_cache"].shape[1], 128,
                                          c["k_cache"].shape[0], c["block_tables"].shape[1]) for c in cases)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    for i, c in enumerate(cases):
        for _ in range(2):
            out = pkv.paged_decode_attention(c["q"], c["k_cache"], c["v_cache"], c["block_tables"],
                                             c["context_lens"], c["scale"], workspace=ws)
            torch.cuda.synchronize()
            assert_attn_close(out, _oracle_rows(c, None), f"shape {i}")


def test_result_independent_of_batch_partition():
    """A sequence's rows do not depend on which other sequences share the launch (each batch
    composition cuts the flattened work differently, so this checks split-count invariance)."""
    lens = [4000, 37, 2500, 900, 16, 3100]
    case = _small_case(lens, hq=16, hkv=4, d=128, seed=51)
    full = _run(case).float().cpu()
    for subset in ([0], [0, 2], [5, 3, 1], [1, 4]):
        idx = torch.tensor(subset)
        sub = {k: (v[idx.to(v.device)] if k in ("q", "block_tables", "context_lens") else v)
               for k, v in case.items()}
        out = _run(sub).float().cpu()
        ref = _oracle_rows(sub, None)
        assert_attn_close(out, ref, f"subset {subset}")
        mx = float((out - full[idx]).abs().max())
        assert mx <= 1e-2, (subset, mx)


def test_cuda_graph_capture_and_replay():
    """The decode calls enqueue no host synchronisation or allocation: captured in a CUDA
    graph and replayed, they give the eager result bit for bit."""
    case = _small_case([700, 33, 1500, 129], hq=8, hkv=2, d=128, seed=52)
    g = torch.Generator().manual_seed(53)
    k_new = rand_bf16((4, 2, 128), g).to(DEV)
    v_new = rand_bf16((4, 2, 128), g).to(DEV)
    ws = torch.zeros(pkv.decode_workspace_bytes(4, 8, 2, 128, case["k_cache"].shape[0],
                                                case["block_tables"].shape[1]), dtype=torch.uint8, device=DEV)
    out = torch.empty_like(case["q"])
    kc0, vc0 = case["k_cache"].clone(), case["v_cache"].clone()
    eager = pkv.paged_decode_attention_append(case["q"], case["k_cache"], case["v_cache"], k_new, v_new,
                                              case["block_tables"], case["context_lens"], case["scale"],
                                              workspace=ws).clone()
    case["k_cache"].copy_(kc0)
    case["v_cache"].copy_(vc0)
    s = torch.cuda.Stream(DEV)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            pkv.paged_decode_attention_append(case["q"], case["k_cache"], case["v_cache"], k_new, v_new,
                                              case["block_tables"], case["context_lens"], case["scale"],
                                              out=out, workspace=ws)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


@pytest.mark.parametrize("seed", range(6))
def test_random_shapes_fuzz(seed):
    """Seeded random shapes: batch, lengths (incl. 0 and block edges), d, G in 1..8, window, and
    the fused append, all against the oracle."""
    rng = np.random.default_rng(1000 + seed)
    d = int(rng.choice([64, 128]))
    hkv = int(rng.integers(1, 5))
    G = int(rng.integers(1, 9))
    B = int(rng.integers(1, 9))
    lens = [int(x) for x in rng.choice([0, 1, 15, 16, 17, 31, 32, 33, 200, 777, 2048, 3000], size=B)]
    window = int(rng.choice([0, 0, 1, 16, 100, 5000]))
    case = _small_case(lens, hq=hkv * G, hkv=hkv, d=d, seed=2000 + seed, fill=float("nan"))
    out = _run(case, window)
    assert_attn_close(out, _oracle_rows(case, None, window=window), f"fuzz {seed}: d={d} G={G} lens={lens}")
    if min(lens) > 0:
        gen = torch.Generator().manual_seed(3000 + seed)
        k_new = rand_bf16((B, hkv, d), gen)
        v_new = rand_bf16((B, hkv, d), gen)
        bt = case["block_tables"].cpu()
        slots = np.array([int(bt[b, (L - 1) // 16]) * 16 + (L - 1) % 16 for b, L in enumerate(lens)],
                         dtype=np.int64)
        okc, ovc = oracle.kv_append(bits(case["k_cache"]), bits(case["v_cache"]), bits(k_new), bits(v_new), slots)
        out2 = pkv.paged_decode_attention_append(case["q"], case["k_cache"], case["v_cache"], k_new.to(DEV),
                                                 v_new.to(DEV), case["block_tables"], case["context_lens"],
                                                 case["scale"], window)
        torch.cuda.synchronize()
        assert np.array_equal(bits(case["k_cache"]), okc) and np.array_equal(bits(case["v_cache"]), ovc)
        assert_attn_close(out2, _oracle_rows(case, None, okc, ovc, window=window), f"fuzz append {seed}")


def _llama8b_ws_case():
    wl = W.WORKLOADS["llama8b"]
    case = W.make_layer(wl, device=DEV, device_rng=True)
    need = pkv.decode_workspace_bytes(wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                      case["num_blocks"], case["max_blocks_per_seq"])
    return wl, case, need


def _decode_ws(case, ws, err=None):
    out = pkv.paged_decode_attention(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                                     case["context_lens"], case["scale"], workspace=ws, error_word=err)
    torch.cuda.synchronize()
    return out


def test_dynamic_tail_chunks_deterministic_rearmed_and_checked():
    """At the llama8b size every worker slice has tail chunks that warps take from a ticket
    counter.  Which warp runs a chunk never changes what it computes, so repeated calls agree
    bit for bit; every call leaves the counters zero; counters that were not zero at the call
    (a workspace not zero-filled) are reported, and the call after that is clean again."""
    wl, case, need = _llama8b_ws_case()
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    err = pkv.new_error_word(DEV)
    outs = [_decode_ws(case, ws, err).clone() for _ in range(3)]
    assert pkv.read_error(err) == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert int(torch.count_nonzero(ws[:8])) == 0
    rows = _sample_rows(wl.batch, wl.num_q_heads, 48, 21)
    ref = _oracle_rows(case, rows)
    assert_attn_close(outs[0].view(-1, wl.head_dim)[torch.tensor(rows, device=DEV)], ref, "llama8b tail chunks")
    dirty = pkv.header_constants()["PKV_DEV_DIRTY_WORKSPACE"]
    for word, value in ((0, 3), (1, 7)):          # a stale ticket count, a stale taken count
        ws[4 * word] = value
        _decode_ws(case, ws, err)
        assert pkv.read_error(err, clear=True) == dirty
        assert int(torch.count_nonzero(ws[:8])) == 0
        again = _decode_ws(case, ws, err)
        assert pkv.read_error(err) == 0
        assert torch.equal(again, outs[0])


def _align256(x):
    return (x + 255) // 256 * 256


def test_smallest_accepted_workspace():
    """A workspace holding the partials of 2048 ranges (static heads only) is accepted and
    gives the same result up to summation order; 256 bytes less is refused."""
    wl, case, need = _llama8b_ws_case()
    B, G, d = wl.batch, wl.num_q_heads // wl.num_kv_heads, wl.head_dim
    slots = 2 * 2048 * G
    ml_off = _align256(256 + 4 * 2 * B)
    smallest = _align256(_align256(ml_off + 8 * slots) + 4 * slots * d)
    assert smallest < need
    full = _decode_ws(case, torch.zeros(need, dtype=torch.uint8, device=DEV)).float()
    err = pkv.new_error_word(DEV)
    out = _decode_ws(case, torch.zeros(smallest, dtype=torch.uint8, device=DEV), err).float()
    assert pkv.read_error(err) == 0
    assert float((out - full).abs().max()) <= 1e-2
    rows = _sample_rows(wl.batch, wl.num_q_heads, 24, 22)
    assert_attn_close(out.view(-1, d)[torch.tensor(rows, device=DEV)], _oracle_rows(case, rows), "smallest ws")
    with pytest.raises(pkv.PkvError) as e:
        _decode_ws(case, torch.zeros(smallest - 256, dtype=torch.uint8, device=DEV))
    assert e.value.status == pkv.header_constants()["PKV_ERR_WORKSPACE"]


def test_large_batch_reads_split_record():
    """Batches above 256 sequences take the merge path that reads the split kernel's record of
    unit starts (smaller ones derive it from the lengths): 320 ragged sequences, some empty,
    enough work for tail chunks."""
    wl = W.Workload("batch320", 91, batch=320, num_q_heads=8, num_kv_heads=2, head_dim=128,
                    len_uniform=(0, 3000))
    lens = W.context_lengths(wl)
    lens[::37] = 0
    case = W.make_layer(wl, device=DEV, lengths=lens, device_rng=True)
    err = pkv.new_error_word(DEV)
    out = _run(case, err=err)
    assert pkv.read_error(err) == 0
    rows = sorted(set(_sample_rows(wl.batch, wl.num_q_heads, 160, 23)) | {37 * 8, 37 * 8 + 7})
    ref = _oracle_rows(case, rows)
    assert_attn_close(out.view(-1, wl.head_dim)[torch.tensor(rows, device=DEV)], ref, "batch 320")
    assert torch.count_nonzero(out[::37]) == 0
