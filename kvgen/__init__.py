"""Seeded synthetic KV-cache inputs shared by the tests, the benchmark and the smoke check.

This module only draws random inputs: BF16 K/V pages with the value distributions of
8B-class models (per-channel scales, outlier channels, injected out-of-window values,
exact zeros, controlled exponent spreads), query vectors, shuffled page tables and
sequence lengths.  It contains none of the compression or attention arithmetic, and
both the CUDA path and the CPU oracle take its outputs as plain inputs.

Layouts (all BF16 pages are [16 tokens][128 dims]):
  raw pool  [num_pages][Hkv][2][16][128]   (2 = K, V)
  q         [B][Hq][128]
  table     [B][pages_per_seq]             physical page ids, a seeded permutation
"""
from __future__ import annotations

import dataclasses

import torch

PAGE = 16
HEAD_DIM = 128


@dataclasses.dataclass(frozen=True)
class KVConfig:
    """Shape and value distribution of one synthetic decode workload."""

    name: str
    layers: int
    batch: int
    hq: int
    hkv: int
    full_pages: int                 # completed (compressible) pages per sequence
    tail_min: int = 0               # tail tokens per sequence drawn in [tail_min, tail_max]
    tail_max: int = 0
    k_log2_sigma: tuple = (-3.0, 2.0)
    v_log2_sigma: tuple = (-3.0, 2.0)
    k_outlier_channels: int = 0     # channels per KV head scaled by k_outlier_scale
    k_outlier_scale: float = 1.0
    block_outlier_frac: float = 0.0  # fraction of blocks with one value set to +-2^block_outlier_log2
    block_outlier_log2: int = 12
    zero_blocks: bool = False       # one all-zero block and one block with a zeroed token row
    spread: tuple | None = None     # per-block exponent spread range (inclusive); replaces N(0, s^2)
    seed: int = 0

    @property
    def pages_per_seq(self) -> int:
        return self.full_pages + (1 if self.tail_max > 0 else 0)

    @property
    def num_pages(self) -> int:
        return self.batch * self.pages_per_seq


# Workloads shaped like the pages' 8B-model decode setups (16-token pages, head dim 128).
C0 = KVConfig("tiny-correctness", layers=1, batch=1, hq=8, hkv=2, full_pages=16,
              k_log2_sigma=(-3, 2), v_log2_sigma=(-3, 2), block_outlier_frac=0.10,
              block_outlier_log2=12, zero_blocks=True, seed=0)
C0_TAIL = dataclasses.replace(C0, name="tiny-correctness-tail", tail_min=7, tail_max=7)
C1 = KVConfig("llama8b-layer-b32-ctx2048", layers=1, batch=32, hq=32, hkv=8, full_pages=128,
              tail_min=1, tail_max=15, k_log2_sigma=(-4, 3), v_log2_sigma=(-3, 1),
              k_outlier_channels=4, k_outlier_scale=32.0, seed=1)
C2 = KVConfig("llama8b-32layer-b16-ctx8192", layers=32, batch=16, hq=32, hkv=8, full_pages=512,
              tail_min=1, tail_max=15, k_log2_sigma=(-4, 3), v_log2_sigma=(-3, 1),
              k_outlier_channels=4, k_outlier_scale=32.0, block_outlier_frac=0.05,
              block_outlier_log2=14, seed=2000)
C3 = KVConfig("qwen3-8b-stream-b64", layers=36, batch=64, hq=32, hkv=8, full_pages=128,
              k_log2_sigma=(-4, 3), v_log2_sigma=(-3, 1), k_outlier_channels=4,
              k_outlier_scale=32.0, seed=3)
C4 = KVConfig("long-ctx-b2-ctx131072", layers=32, batch=2, hq=32, hkv=8, full_pages=8192,
              tail_min=1, tail_max=15, spread=(8, 20), seed=4)

CONFIGS = {"c0": C0, "c0t": C0_TAIL, "c1": C1, "c2": C2, "c3": C3, "c4": C4}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _uniform(g, shape, lo, hi, device):
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def channel_sigmas(cfg: KVConfig, layer: int, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """Per-(KV head, channel) standard deviations for K and V, each [Hkv][128]."""
    g = _gen(device, cfg.seed * 1000003 + layer * 7919 + 17)
    ks = torch.exp2(_uniform(g, (cfg.hkv, HEAD_DIM), *cfg.k_log2_sigma, device))
    vs = torch.exp2(_uniform(g, (cfg.hkv, HEAD_DIM), *cfg.v_log2_sigma, device))
    if cfg.k_outlier_channels:
        for h in range(cfg.hkv):
            idx = torch.randperm(HEAD_DIM, generator=g, device=device)[: cfg.k_outlier_channels]
            ks[h, idx] *= cfg.k_outlier_scale
    return ks, vs


def gen_pages(cfg: KVConfig, num_pages: int, layer: int = 0, device="cpu", seed_offset: int = 0) -> torch.Tensor:
    """BF16 raw pool [num_pages][Hkv][2][16][128] for one layer."""
    g = _gen(device, cfg.seed * 7777 + layer * 131 + seed_offset + 1)
    shape = (num_pages, cfg.hkv, 2, PAGE, HEAD_DIM)
    if cfg.spread is not None:
        return _spread_pages(cfg, g, num_pages, device)
    ks, vs = channel_sigmas(cfg, layer, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    x[:, :, 0] *= ks[None, :, None, :]
    x[:, :, 1] *= vs[None, :, None, :]
    pool = x.to(torch.bfloat16)
    del x
    # a block is one (page, head, K|V) slab of 16 tokens x 32 dims
    blocks = pool.view(num_pages, cfg.hkv, 2, PAGE, 4, 32)
    nblk = num_pages * cfg.hkv * 2 * 4
    if cfg.block_outlier_frac > 0:
        pick = torch.rand(nblk, generator=g, device=device) < cfg.block_outlier_frac
        ids = torch.nonzero(pick).flatten()
        if ids.numel():
            tok = torch.randint(0, PAGE, (ids.numel(),), generator=g, device=device)
            col = torch.randint(0, 32, (ids.numel(),), generator=g, device=device)
            sgn = torch.randint(0, 2, (ids.numel(),), generator=g, device=device).float() * 2 - 1
            j = ids % 4
            rest = ids // 4
            kv = rest % 2
            rest = rest // 2
            h = rest % cfg.hkv
            p = rest // cfg.hkv
            val = (sgn * float(2 ** cfg.block_outlier_log2)).to(torch.bfloat16)
            blocks[p, h, kv, tok, j, col] = val
    if cfg.zero_blocks and num_pages >= 2:
        # one block entirely +0, and one block whose token-3 row is zero (mixed signs)
        blocks[0, 0, 0, :, 1, :] = 0
        row = torch.zeros(32, dtype=torch.bfloat16, device=device)
        row[::2] = -0.0
        blocks[1, cfg.hkv - 1, 1, 3, 2, :] = row
    return pool


_SPREAD_CHUNK = 1 << 18  # blocks generated per chunk (bounds the temporaries to ~0.5 GB)


def _spread_pages(cfg: KVConfig, g, num_pages: int, device) -> torch.Tensor:
    """Per block: spread S ~ U{lo..hi}; exponents uniform in [E0, E0+S] with both ends
    present, E0 = 127 - S + (random parity bit); random sign and fraction."""
    lo, hi = cfg.spread
    nblk = num_pages * cfg.hkv * 2 * 4
    words = torch.empty((nblk, 512), dtype=torch.int16, device=device)
    for b0 in range(0, nblk, _SPREAD_CHUNK):
        n = min(_SPREAD_CHUNK, nblk - b0)
        S = torch.randint(lo, hi + 1, (n, 1), generator=g, device=device, dtype=torch.int32)
        E0 = 127 - S + torch.randint(0, 2, (n, 1), generator=g, device=device, dtype=torch.int32)
        u = torch.rand((n, 512), generator=g, device=device)
        e = torch.minimum(E0 + torch.floor(u * (S + 1).float()).to(torch.int32), E0 + S)
        del u
        # force both ends of the window to occur
        pos = torch.randint(0, 512, (n, 2), generator=g, device=device)
        pos[:, 1] = (pos[:, 0] + 1 + torch.randint(0, 511, (n,), generator=g, device=device)) % 512
        e.scatter_(1, pos[:, :1], E0)
        e.scatter_(1, pos[:, 1:], E0 + S)
        sign = torch.randint(0, 2, (n, 512), generator=g, device=device, dtype=torch.int32)
        frac = torch.randint(0, 128, (n, 512), generator=g, device=device, dtype=torch.int32)
        w = (sign << 15) | (e << 7) | frac
        del sign, frac, e
        words[b0: b0 + n] = torch.where(w >= 32768, w - 65536, w).to(torch.int16)
        del w
    # block order (page, head, kv, j) with values [16 tok][32 dims] -> page layout
    w = words.view(num_pages, cfg.hkv, 2, 4, PAGE, 32).permute(0, 1, 2, 4, 3, 5).contiguous()
    return w.view(num_pages, cfg.hkv, 2, PAGE, HEAD_DIM).view(torch.bfloat16)


def gen_new_tokens(cfg: KVConfig, steps: int, device="cpu") -> torch.Tensor:
    """K/V of the tokens appended during `steps` decode steps, all layers:
    BF16 [steps][layers][B][Hkv][2][128], same per-channel scales as the prompt pages."""
    out = torch.empty((steps, cfg.layers, cfg.batch, cfg.hkv, 2, HEAD_DIM), dtype=torch.bfloat16, device=device)
    for layer in range(cfg.layers):
        ks, vs = channel_sigmas(cfg, layer, device)
        g = _gen(device, cfg.seed * 4241 + layer * 97 + 11)
        x = torch.randn((steps, cfg.batch, cfg.hkv, 2, HEAD_DIM), generator=g, device=device)
        x[:, :, :, 0] *= ks[None, None]
        x[:, :, :, 1] *= vs[None, None]
        out[:, layer] = x.to(torch.bfloat16)
    return out


def gen_q(cfg: KVConfig, layer: int = 0, device="cpu", step: int = 0) -> torch.Tensor:
    g = _gen(device, cfg.seed * 31 + layer * 1009 + step * 65537 + 5)
    return torch.randn((cfg.batch, cfg.hq, HEAD_DIM), generator=g, device=device).to(torch.bfloat16)


def gen_layout(cfg: KVConfig, device="cpu") -> dict:
    """Page table and lengths for one layer.

    table[b] lists sequence b's physical pages in order (the last column is the tail
    page when tails are enabled); tail_len[b] is the number of tail tokens.  Returns
    table [B][pages_per_seq], seq_lens [B], tail_len [B]."""
    g = _gen("cpu", cfg.seed * 13 + 3)
    perm = torch.randperm(cfg.num_pages, generator=g).to(torch.int32)
    table = perm.view(cfg.batch, cfg.pages_per_seq)
    if cfg.tail_max > 0:
        tail = torch.randint(cfg.tail_min, cfg.tail_max + 1, (cfg.batch,), generator=g).to(torch.int32)
    else:
        tail = torch.zeros(cfg.batch, dtype=torch.int32)
    seq_lens = (cfg.full_pages * PAGE + tail).to(torch.int32)
    return {
        "table": table.to(device),
        "seq_lens": seq_lens.to(device),
        "tail_len": tail.to(device),
    }


def bits(t: torch.Tensor):
    """BF16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    import numpy as np

    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def logical_kv_bytes(cfg: KVConfig, seq_lens) -> int:
    """BF16 bytes of K and V attended per layer (tokens x Hkv x 2 x 128 x 2 B)."""
    total_tokens = int(torch.as_tensor(seq_lens).sum())
    return total_tokens * cfg.hkv * 2 * HEAD_DIM * 2

