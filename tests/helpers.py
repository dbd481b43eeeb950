"""Test-side helpers: tensor <-> oracle marshalling and contiguous -> paged construction.

The paged construction here scatters a contiguous K/V array into a shuffled pool by the
pool layout the library documents ([NB, Hkv, 16, d], token t of sequence b at block
block_tables[b][t // 16], offset t % 16).  Tests use it to build cases whose expected
result is known from the contiguous data, independently of the oracle's gather.
"""
import numpy as np
import torch

BLOCK = 16


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 of its raw bits (on the host)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def stored_codes(codes) -> np.ndarray:
    """INT8 codes (integers in [-128, 127]) as the pools store them: the byte code + 128."""
    return (np.asarray(codes, dtype=np.int32) + 128).astype(np.uint8)


def code_values(stored) -> np.ndarray:
    """The INT8 codes of stored pool bytes (numpy or torch): byte - 128, as int32."""
    if isinstance(stored, torch.Tensor):
        stored = stored.cpu().numpy()
    return np.asarray(stored).astype(np.int32) - 128


def rand_code_pool(shape, gen, device=None) -> torch.Tensor:
    """A pool of random INT8 codes in [-127, 127], stored as bytes code + 128 (uint8)."""
    return torch.randint(1, 256, shape, generator=gen, device=device, dtype=torch.uint8)


def paged_from_contiguous(k, v, lens, num_blocks, gen, max_blocks=None, fill=None):
    """Scatter contiguous k, v [B, Lmax, Hkv, d] (bf16) into shuffled pools.

    Returns (k_cache, v_cache, block_tables) with pools [NB, Hkv, 16, d] bf16; unused pool
    rows hold N(0,1) noise (or `fill`, e.g. NaN, to catch reads past the context).
    """
    B, lmax, hkv, d = k.shape
    nblk = [(int(L) + BLOCK - 1) // BLOCK for L in lens]
    mb = max(nblk + [1]) if max_blocks is None else max_blocks
    perm = torch.randperm(num_blocks, generator=gen)
    if fill is None:
        kc = torch.randn((num_blocks, hkv, BLOCK, d), generator=gen).to(torch.bfloat16)
        vc = torch.randn((num_blocks, hkv, BLOCK, d), generator=gen).to(torch.bfloat16)
    else:
        kc = torch.full((num_blocks, hkv, BLOCK, d), fill, dtype=torch.bfloat16)
        vc = torch.full((num_blocks, hkv, BLOCK, d), fill, dtype=torch.bfloat16)
    bt = torch.full((B, mb), -1, dtype=torch.int32)
    off = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[off:off + nblk[b]].to(torch.int32)
        off += nblk[b]
        for t in range(int(lens[b])):
            blk = int(bt[b, t // BLOCK])
            kc[blk, :, t % BLOCK, :] = k[b, t]
            vc[blk, :, t % BLOCK, :] = v[b, t]
    return kc, vc, bt


def rand_bf16(shape, gen):
    return torch.randn(shape, generator=gen).to(torch.bfloat16)


# Tolerance of the floating-point parity gate: bf16 inputs, fp32 accumulation, bf16 output,
# compared with the fp64 oracle.
MAX_ABS = 1e-2
REL_L2 = 2e-3


def attn_errors(got: torch.Tensor, ref: np.ndarray):
    """(max-abs, relative L2) of a bf16 GPU result against the fp64 oracle."""
    g = got.detach().float().cpu().double().numpy().reshape(ref.shape)
    diff = g - ref
    denom = np.linalg.norm(ref)
    rel = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    return float(np.abs(diff).max()) if diff.size else 0.0, rel


def assert_attn_close(got: torch.Tensor, ref: np.ndarray, what: str = ""):
    mx, rel = attn_errors(got, ref)
    assert np.all(np.isfinite(got.detach().float().cpu().numpy())), f"{what}: non-finite output"
    assert mx <= MAX_ABS and rel <= REL_L2, f"{what}: max-abs {mx:.3e} rel-L2 {rel:.3e}"
    return mx, rel
