"""The seeded workload generators: deterministic, and shaped as the workloads state."""
import torch

from paged_kv_cache_mapped_gb300 import inputs as W


def test_lengths_follow_recipes():
    assert W.context_lengths(W.WORKLOADS["tiny"]).tolist() == [100, 256]
    l2 = W.context_lengths(W.WORKLOADS["llama8b"])
    assert l2.shape == (32,) and int(l2.min()) >= 3501 and int(l2.max()) <= 4501
    l3 = W.context_lengths(W.WORKLOADS["qwen1p5b"])
    assert l3.shape == (64,) and int(l3.min()) >= 16 and int(l3.max()) <= 4096
    assert 1200 < float(l3.float().median()) < 3200
    assert W.context_lengths(W.WORKLOADS["long128k"]).tolist() == [131072] * 4
    assert W.context_lengths(W.WORKLOADS["sparse"]).tolist() == [16384] * 16


def test_layer_is_deterministic_and_tables_valid():
    wl = W.WORKLOADS["tiny"]
    a = W.make_layer(wl)
    b = W.make_layer(wl)
    for key in ("q", "k_cache", "v_cache", "block_tables", "context_lens"):
        assert torch.equal(a[key].view(torch.int16) if a[key].dtype == torch.bfloat16 else a[key],
                           b[key].view(torch.int16) if b[key].dtype == torch.bfloat16 else b[key])
    bt = a["block_tables"]
    used = bt[bt >= 0]
    assert used.numel() == 7 + 16 and used.unique().numel() == used.numel()
    assert int(used.max()) < a["num_blocks"] == 64
    c = W.make_layer(wl, layer=1)
    assert not torch.equal(a["k_cache"].view(torch.int16), c["k_cache"].view(torch.int16))


def test_append_slot_is_last_position():
    wl = W.WORKLOADS["llama8b"]
    lens = torch.tensor([17, 16, 1], dtype=torch.int32)
    case = W.make_layer(wl, lengths=lens)
    bt, slot = case["block_tables"], case["slot_mapping"]
    for b, L in enumerate(lens.tolist()):
        assert int(slot[b]) // 16 == int(bt[b, (L - 1) // 16])
        assert int(slot[b]) % 16 == (L - 1) % 16


def test_sink_keys_scaled():
    wl = W.WORKLOADS["long128k"]
    lens = torch.tensor([40, 40, 40, 40], dtype=torch.int32)
    case = W.make_layer(wl, lengths=lens, num_blocks=16)
    kc, bt = case["k_cache"].float(), case["block_tables"]
    blk = int(bt[0, 0])
    sink_rms = kc[blk, :, :2].pow(2).mean().sqrt()
    rest_rms = kc[blk, :, 2:].pow(2).mean().sqrt()
    assert sink_rms > 10 * rest_rms


def test_scores_exponential():
    wl = W.WORKLOADS["sparse"]
    s = W.make_scores(wl, 4, torch.tensor([1000, 1000], dtype=torch.int32))
    assert s.shape == (2, 8, 1000) and s.dtype == torch.float32
    assert float(s.min()) >= 0.0 and 0.9 < float(s.mean()) < 1.1
