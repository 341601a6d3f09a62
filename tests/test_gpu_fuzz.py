"""Seeded random shapes for the decode-attention path (ZipFusion "How it works"; GAAC
"Attention with On-the-Fly Decompression"): batch, KV heads, group size, context,
per-sequence lengths (empty, tail-only, page multiples, arbitrary), value distributions
and launch mode drawn per case.  Each case: the GPU encoder's bytes, metadata and cursors
against the oracle's bit for bit; the compressed and the raw kernel against the fp64
oracle within the attention tolerance, and against each other bit for bit."""
import numpy as np
import pytest
import torch

import kvgen
from helpers import F8Layer, GaLayer, Layer, check_attention

pytestmark = pytest.mark.gpu

N_CASES = 24


@pytest.fixture(scope="module")
def kvz():
    from decode_attention_value_gb300 import _build

    _build.build()
    import decode_attention_value_gb300 as m

    return m


def _case(i: int):
    rng = np.random.default_rng(9000 + i)
    hkv = int(rng.choice([1, 2, 4, 8, 16]))
    G = int(rng.integers(1, 9))
    batch = int(rng.integers(1, 41))
    full = int(rng.integers(0, 33))
    tail = bool(rng.integers(0, 4))  # a tail column in three cases of four
    dist = int(rng.integers(0, 3))
    kw = {}
    if dist == 0:  # Gaussian channels with outlier channels and outlier blocks
        kw = dict(k_log2_sigma=(-4, 3), v_log2_sigma=(-3, 1), k_outlier_channels=int(rng.integers(0, 5)),
                  k_outlier_scale=32.0, block_outlier_frac=float(rng.choice([0.0, 0.05, 0.3])),
                  block_outlier_log2=int(rng.choice([12, 14])), zero_blocks=bool(rng.integers(0, 2)))
    elif dist == 1:  # per-block exponent spreads around the eligibility limit
        lo = int(rng.integers(8, 16))
        kw = dict(spread=(lo, int(rng.integers(lo, 21))))
    else:  # narrow or wide Gaussians
        s = float(rng.choice([-6.0, 0.0, 4.0]))
        kw = dict(k_log2_sigma=(s - 1, s + 1), v_log2_sigma=(s - 2, s))
    cfg = kvgen.KVConfig(f"fuzz{i}", 1, batch, hkv * G, hkv, full, tail_min=1 if tail else 0,
                         tail_max=15 if tail else 0, seed=9100 + i, **kw)
    # lengths: full pages fill the table's compressed columns; a partial last page (at most
    # 15 tokens) needs the tail column, so without it whole pages only
    cap = full * kvgen.PAGE + (kvgen.PAGE - 1 if tail else 0)
    kind = rng.integers(0, 4, batch)
    lens = []
    for b in range(batch):
        if kind[b] == 0:
            L = 0
        elif kind[b] == 1 and tail:
            L = int(rng.integers(1, 16))  # tail only
        elif kind[b] == 2:
            L = kvgen.PAGE * int(rng.integers(0, full + 1))
        else:
            L = int(rng.integers(0, cap + 1))
        if not tail:
            L -= L % kvgen.PAGE
        lens.append(min(L, cap))
    flags = int(rng.integers(0, 2))
    return cfg, lens, flags


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shapes_match_oracle(kvz, oracle, i):
    cfg, lens, flags = _case(i)
    layer = Layer(cfg, oracle, seq_lens=lens)
    # the encoder's pages, metadata and cursors bit for bit
    assert np.array_equal(layer.meta.cpu().numpy().view(np.uint64), layer.o_meta), f"{cfg.name}: metadata"
    assert np.array_equal(layer.arena.cpu().numpy(), layer.o_arena), f"{cfg.name}: arena bytes"
    assert np.array_equal(layer.cursors.cpu().numpy().view(np.uint32), layer.o_cursors), f"{cfg.name}: cursors"
    out_c = layer.run_compressed(flags=flags)
    out_r = layer.run_raw(flags=flags)
    torch.cuda.synchronize()
    what = f"{cfg.name} (B={cfg.batch}, Hkv={cfg.hkv}, G={cfg.hq // cfg.hkv}, pages={cfg.full_pages}, flags={flags})"
    assert int(layer.status.item()) == 0, f"{what}: status {int(layer.status.item())}"
    ref, st = layer.oracle_attention(oracle)
    assert st == 0
    check_attention(out_c, ref, what + " compressed")
    check_attention(out_r, ref, what + " raw")
    assert torch.equal(out_c, out_r), f"{what}: compressed and raw outputs differ"
    empty = [b for b, L in enumerate(lens) if L == 0]
    if empty:
        assert not out_c[empty].any(), f"{what}: empty sequences must give zero outputs"


def _u32(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("i", range(8))
def test_random_shapes_group_adaptive_tiles(kvz, oracle, i):
    """The group-adaptive tile format on the same random draws: calibration bases, tile
    entries and bytes and cursors bit for bit, attention within the tolerance of the fp64
    oracle and bit-identical to the raw kernel."""
    cfg, lens, _ = _case(100 + i)
    base = Layer(cfg, None, seq_lens=lens)
    ga = GaLayer(base, oracle)
    what = f"{cfg.name} tiles (B={cfg.batch}, Hkv={cfg.hkv}, G={cfg.hq // cfg.hkv}, pages={cfg.full_pages})"
    assert np.array_equal(ga.bases.cpu().numpy(), ga.o_bases), what + ": bases"
    assert np.array_equal(_u32(ga.meta), ga.o_meta), what + ": entries"
    assert np.array_equal(ga.arena.cpu().numpy(), ga.o_arena), what + ": tile bytes"
    assert np.array_equal(_u32(ga.cursors), ga.o_cursors), what + ": cursors"
    out_g = ga.run()
    out_r = base.run_raw()
    torch.cuda.synchronize()
    assert int(ga.status.item()) == 0 and int(base.status.item()) == 0, what
    ref, st = ga.oracle_attention(oracle)
    assert st == 0
    check_attention(out_g, ref, what)
    assert torch.equal(out_g, out_r), what + ": tile and raw outputs differ"


@pytest.mark.parametrize("fmt", [1, 2], ids=["e4m3", "e5m2"])
@pytest.mark.parametrize("i", range(4))
def test_random_shapes_fp8_tiles(kvz, oracle, fmt, i):
    """FP8 pages on the same random draws: bases, entries, tile bytes and cursors bit for
    bit, attention within the tolerance of the fp64 oracle over the FP8 values."""
    cfg, lens, _ = _case(200 + i)
    base = Layer(cfg, None, seq_lens=lens)
    f8 = F8Layer(base, fmt, oracle)
    what = f"{cfg.name} fp8 {fmt} (B={cfg.batch}, Hkv={cfg.hkv}, G={cfg.hq // cfg.hkv}, pages={cfg.full_pages})"
    assert np.array_equal(f8.bases.cpu().numpy(), f8.o_bases), what + ": bases"
    assert np.array_equal(_u32(f8.meta), f8.o_meta), what + ": entries"
    assert np.array_equal(f8.arena.cpu().numpy(), f8.o_arena), what + ": tile bytes"
    assert np.array_equal(_u32(f8.cursors), f8.o_cursors), what + ": cursors"
    got = f8.run()
    torch.cuda.synchronize()
    assert int(f8.status.item()) == 0, what
    ref, st = f8.oracle_attention(oracle)
    assert st == 0
    check_attention(got, ref, what)
