"""Seeded synthetic workloads for paged decode attention.

This module only draws inputs: context lengths, shuffled block tables, q, the K/V pools,
the new token's K/V with its slot, and accumulated scores for the sparse layers.  It holds
none of the attention, selection or compaction arithmetic, so the CUDA library and the
fp64 oracle can both be fed from it without sharing any of the method.

Recipe (all draws from one seeded ``torch.Generator`` per workload and layer):
  * lengths: fixed, uniform integer, or log-normal (median, sigma in log space, clipped);
    L_b counts the token appended this step; every layer of a step shares them.
  * pool: NB physical blocks (fixed, or ceil(1.1 x blocks needed)); the blocks of all
    sequences are the first sum_b ceil(L_b/16) entries of a random permutation of the pool,
    handed out in sequence order; unused table entries are -1.
  * q, K, V, new K/V: N(0,1) drawn in fp32 and rounded to bf16 (round-to-nearest-even).
    Optional sink positions get K = bf16(scale * N(0,1)) on every kv head.
  * scores: Exp(1) fp32.
  * the appended token of sequence b sits at logical position L_b - 1; its slot is the
    physical position the block manager assigned to it (block table entry * 16 + offset).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BLOCK_SIZE = 16
BASE_SEED = 20261202


@dataclass(frozen=True)
class Workload:
    name: str
    index: int                 # 1-based workload number; the seed is BASE_SEED + index
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    layers: int = 1
    lengths: tuple = ()        # fixed lengths (cycled over the batch) when non-empty
    len_uniform: tuple = ()    # (lo, hi) inclusive prefix length; L = prefix + 1
    len_lognormal: tuple = ()  # (median, sigma, lo, hi)
    pool_blocks: int = 0       # fixed pool size; 0 -> ceil(1.1 * needed)
    sink_positions: int = 0    # leading positions whose K is scaled
    sink_scale: float = 1.0
    append: bool = False       # the step appends one token per sequence first
    full_layers: int = -1      # sparse workloads: layers [0, full_layers) keep the full cache
    n_sink: int = 0
    n_recent: int = 0
    k_top: int = 0
    notes: str = field(default="", compare=False)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def keep_max(self) -> int:
        return self.n_sink + self.k_top + self.n_recent

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


WORKLOADS = {
    "tiny": Workload("tiny", 1, batch=2, num_q_heads=8, num_kv_heads=8, head_dim=64,
                     lengths=(100, 256), pool_blocks=64,
                     notes="tiny paged decode, parity only"),
    "llama8b": Workload("llama8b", 2, batch=32, num_q_heads=32, num_kv_heads=8, head_dim=128,
                        len_uniform=(3500, 4500), append=True,
                        notes="Llama-3-8B-shaped decode layer, ~4000-in/500-out serving shape"),
    "qwen1p5b": Workload("qwen1p5b", 3, batch=64, num_q_heads=12, num_kv_heads=2, head_dim=128,
                         layers=28, len_lognormal=(2048.0, 0.5, 16, 4096), append=True,
                         notes="Qwen2.5-1.5B-shaped full decode step, separate pool per layer"),
    "long128k": Workload("long128k", 4, batch=4, num_q_heads=32, num_kv_heads=8, head_dim=128,
                         lengths=(131072,), pool_blocks=32768, sink_positions=2, sink_scale=20.0,
                         notes="long-context split-K decode with two 20x sink keys"),
    "sparse": Workload("sparse", 5, batch=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
                       layers=32, lengths=(16384,), full_layers=4, n_sink=4, n_recent=1024,
                       k_top=512, notes="layer-wise sparse decode"),
}


def _cpu_gen(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(seed)


def layer_seed(wl: Workload, layer: int, salt: int = 0) -> int:
    return BASE_SEED + wl.index + 7919 * layer + 104729 * salt


def context_lengths(wl: Workload, batch: int | None = None) -> torch.Tensor:
    """int32 [B] context lengths (including the token appended this step)."""
    b = wl.batch if batch is None else batch
    g = _cpu_gen(BASE_SEED + wl.index)
    if wl.lengths:
        vals = [wl.lengths[i % len(wl.lengths)] for i in range(b)]
        return torch.tensor(vals, dtype=torch.int32)
    if wl.len_uniform:
        lo, hi = wl.len_uniform
        prefix = torch.randint(lo, hi + 1, (b,), generator=g, dtype=torch.int64)
        return (prefix + 1).to(torch.int32)
    if wl.len_lognormal:
        median, sigma, lo, hi = wl.len_lognormal
        z = torch.randn((b,), generator=g, dtype=torch.float64)
        vals = torch.exp(math.log(median) + sigma * z).round().clamp(lo, hi)
        return vals.to(torch.int32)
    raise ValueError(f"workload {wl.name} has no length recipe")


def blocks_needed(lengths: torch.Tensor) -> torch.Tensor:
    return (lengths.to(torch.int64) + BLOCK_SIZE - 1) // BLOCK_SIZE


def block_tables_for(lengths: torch.Tensor, num_blocks: int, max_blocks: int,
                     gen: torch.Generator) -> torch.Tensor:
    """int32 [B, max_blocks]: sequence b owns consecutive entries of a pool permutation."""
    nblk = blocks_needed(lengths)
    total = int(nblk.sum())
    if total > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {total}")
    perm = torch.randperm(num_blocks, generator=gen).to(torch.int32)
    bt = torch.full((lengths.shape[0], max_blocks), -1, dtype=torch.int32)
    off = 0
    for b in range(lengths.shape[0]):
        n = int(nblk[b])
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt


def _randn_bf16(shape, gen: torch.Generator, device, chunk_elems: int = 1 << 26) -> torch.Tensor:
    """N(0,1) in fp32 rounded to bf16, drawn in chunks along dim 0 to bound fp32 memory."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1) if len(shape) > 1 else out.view(-1, 1)
    row = flat.shape[1]
    step = max(1, chunk_elems // max(row, 1))
    for s in range(0, flat.shape[0], step):
        e = min(flat.shape[0], s + step)
        flat[s:e] = torch.randn((e - s, row), generator=gen, device=device,
                                dtype=torch.float32).to(torch.bfloat16)
    return out


def pool_size(wl: Workload, lengths: torch.Tensor) -> int:
    if wl.pool_blocks:
        return wl.pool_blocks
    return int(math.ceil(1.1 * int(blocks_needed(lengths).sum())))


def make_layer(wl: Workload, layer: int = 0, device="cpu", lengths: torch.Tensor | None = None,
               device_rng: bool = False, max_blocks: int | None = None,
               num_blocks: int | None = None) -> dict:
    """One layer's decode inputs.

    Returns a dict of tensors on `device`: q [B,Hq,d], k_cache/v_cache [NB,Hkv,16,d] bf16,
    block_tables [B,MB] int32, context_lens [B] int32; with wl.append also k_new/v_new
    [B,Hkv,d] bf16 and slot_mapping [B] int64.  Lengths, permutation and slots always come
    from the CPU generator; with device_rng the large N(0,1) tensors are drawn by a seeded
    generator on `device` instead (fast for multi-GB pools; a different but equally seeded
    stream).  num_blocks overrides the workload's pool size (small test cases).
    """
    lens = context_lengths(wl) if lengths is None else lengths.to(torch.int32).cpu()
    nb = pool_size(wl, lens) if num_blocks is None else num_blocks
    mb = int(blocks_needed(lens).max()) if max_blocks is None else max_blocks
    seed = layer_seed(wl, layer)
    cpu_g = _cpu_gen(seed)
    bt = block_tables_for(lens, nb, mb, cpu_g)
    dev = torch.device(device)
    if device_rng and dev.type != "cpu":
        rg = torch.Generator(device=dev).manual_seed(seed)
        rdev = dev
    else:
        rg = cpu_g
        rdev = torch.device("cpu")
    B, hq, hkv, d = lens.shape[0], wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    q = _randn_bf16((B, hq, d), rg, rdev)
    kc = _randn_bf16((nb, hkv, BLOCK_SIZE, d), rg, rdev)
    vc = _randn_bf16((nb, hkv, BLOCK_SIZE, d), rg, rdev)
    if wl.sink_positions:
        sinks = torch.randn((B, hkv, wl.sink_positions, d), generator=rg, device=rdev,
                            dtype=torch.float32)
        sinks = (sinks * wl.sink_scale).to(torch.bfloat16)
        for b in range(B):
            for p in range(min(wl.sink_positions, int(lens[b]))):
                blk = int(bt[b, p // BLOCK_SIZE])
                kc[blk, :, p % BLOCK_SIZE, :] = sinks[b, :, p, :]
    case = {
        "workload": wl.name,
        "layer": layer,
        "q": q.to(dev),
        "k_cache": kc.to(dev),
        "v_cache": vc.to(dev),
        "block_tables": bt.to(dev),
        "context_lens": lens.to(dev),
        "scale": wl.scale,
        "num_blocks": nb,
        "max_blocks_per_seq": mb,
    }
    if wl.append:
        k_new = _randn_bf16((B, hkv, d), rg, rdev)
        v_new = _randn_bf16((B, hkv, d), rg, rdev)
        pos = lens.to(torch.int64) - 1
        slot = torch.full((B,), -1, dtype=torch.int64)
        for b in range(B):
            if pos[b] >= 0:
                slot[b] = int(bt[b, int(pos[b]) // BLOCK_SIZE]) * BLOCK_SIZE + int(pos[b]) % BLOCK_SIZE
        case.update(k_new=k_new.to(dev), v_new=v_new.to(dev), slot_mapping=slot.to(dev))
    return case


def make_scores(wl: Workload, layer: int, lengths: torch.Tensor, device="cpu",
                device_rng: bool = False) -> torch.Tensor:
    """Accumulated attention scores ~ Exp(1) fp32 [B, Hkv, max L] for one sparse layer."""
    lmax = int(lengths.max())
    shape = (lengths.shape[0], wl.num_kv_heads, lmax)
    dev = torch.device(device)
    seed = layer_seed(wl, layer, salt=1)
    if device_rng and dev.type != "cpu":
        g = torch.Generator(device=dev).manual_seed(seed)
        return torch.empty(shape, dtype=torch.float32, device=dev).exponential_(generator=g)
    g = _cpu_gen(seed)
    return torch.empty(shape, dtype=torch.float32).exponential_(generator=g).to(dev)


def compact_tables(kept_lens_max: int, batch: int, num_blocks: int | None = None,
                   seed: int = BASE_SEED) -> tuple[torch.Tensor, int]:
    """Block tables of a destination pool for compacted sparse layers (shuffled, like vLLM)."""
    per_seq = (kept_lens_max + BLOCK_SIZE - 1) // BLOCK_SIZE
    lens = torch.full((batch,), per_seq * BLOCK_SIZE, dtype=torch.int32)
    nb = batch * per_seq if num_blocks is None else num_blocks
    return block_tables_for(lens, nb, per_seq, _cpu_gen(seed)), nb
