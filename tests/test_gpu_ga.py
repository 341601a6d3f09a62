"""GPU parity of the group-adaptive additive tile format (GAAC, "Lossless KV
Compression" and "Attention with On-the-Fly Decompression"): calibrated bases, tile
bytes and entries bit-exact against the CPU oracle, bit-exact standalone decode, and
attention within the stated tolerance of the fp64 oracle and bit-identical to the raw
kernel."""
import numpy as np
import pytest
import torch

import kvgen
from helpers import GaLayer, Layer, check_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvz():
    from decode_attention_value_gb300 import _build

    _build.build()
    import decode_attention_value_gb300 as m

    return m


CASES = [
    kvgen.C0,
    kvgen.C0_TAIL,
    kvgen.KVConfig("ragged-b6", 1, 6, 16, 4, 9, tail_min=1, tail_max=15, k_log2_sigma=(-4, 3),
                   v_log2_sigma=(-3, 1), k_outlier_channels=4, k_outlier_scale=32.0, block_outlier_frac=0.05,
                   block_outlier_log2=14, seed=31),
    kvgen.KVConfig("gqa1", 1, 3, 4, 4, 7, tail_min=3, tail_max=9, seed=32),
    kvgen.KVConfig("gqa2", 1, 3, 8, 4, 7, tail_min=3, tail_max=9, seed=33),
    kvgen.KVConfig("gqa8", 1, 5, 16, 2, 11, tail_min=1, tail_max=15, k_log2_sigma=(-4, 3), v_log2_sigma=(-3, 1),
                   seed=36),
    # wide exponent spreads: many 4-bit and raw groups, some tiles fall back to raw
    kvgen.KVConfig("spread", 1, 2, 32, 8, 12, tail_min=1, tail_max=15, spread=(6, 12), seed=34),
    kvgen.KVConfig("gqa3", 1, 3, 6, 2, 7, tail_min=1, tail_max=15, k_log2_sigma=(-4, 3), seed=38),
    kvgen.KVConfig("gqa6", 1, 3, 12, 2, 9, tail_min=1, tail_max=15, v_log2_sigma=(-3, 1), seed=40),
    kvgen.KVConfig("llama-b4", 1, 4, 32, 8, 20, tail_min=1, tail_max=15, k_log2_sigma=(-4, 3),
                   v_log2_sigma=(-3, 1), k_outlier_channels=4, k_outlier_scale=32.0, seed=35),
]


def _np_meta(t):
    return t.cpu().numpy().view(np.uint32)


def _check_codec(ga, what):
    assert np.array_equal(ga.bases.cpu().numpy(), ga.o_bases), f"{what}: bases differ"
    assert np.array_equal(_np_meta(ga.meta), ga.o_meta), f"{what}: entries differ"
    assert np.array_equal(ga.arena.cpu().numpy(), ga.o_arena), f"{what}: tile bytes differ"
    assert np.array_equal(ga.cursors.cpu().numpy().view(np.uint32), ga.o_cursors), f"{what}: cursors differ"


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_codec_and_attention(kvz, oracle, cfg):
    base = Layer(cfg, None)
    ga = GaLayer(base, oracle)
    _check_codec(ga, cfg.name)
    # standalone decode returns the input bits
    if base.src.numel():
        out = torch.empty((base.src.numel(), cfg.hkv, 2, 16, 128), dtype=torch.bfloat16, device="cuda")
        st = kvz.new_status()
        kvz.ga_decode_blocks(ga.meta, ga.arena, ga.bases, base.src.cuda(), out, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(out.view(torch.int16), base.g_pool[base.src.cuda().long()].view(torch.int16))
    # attention: oracle tolerance, and bit-identical to the raw kernel
    out_g = ga.run()
    out_r = base.run_raw()
    torch.cuda.synchronize()
    assert int(ga.status.item()) == 0 and int(base.status.item()) == 0
    ref, st = ga.oracle_attention(oracle)
    assert st == 0
    check_attention(out_g, ref, cfg.name + " tiles")
    assert torch.equal(out_g, out_r), f"{cfg.name}: tile and raw outputs differ"


def _tile_modes(ga):
    meta = _np_meta(ga.meta)[ga.base.src.numpy()].reshape(-1)
    raw = (meta & 0x80000000) != 0
    arena = ga.arena.cpu().numpy()
    modes = np.zeros(4, np.int64)
    for e in meta[~raw]:
        tags = arena[int(e) * 64 + 2816: int(e) * 64 + 2880]
        for s in range(0, 8, 2):
            modes += np.bincount((tags >> s) & 3, minlength=4)
    return raw, modes


def test_mode_mix_is_exercised(kvz, oracle):
    """The cases above hold every group mode inside compressed tiles and both tile
    classes: wide spreads overflow the escape slot, injected outliers need raw groups."""
    by_name = {c.name: c for c in CASES}
    raw, modes = _tile_modes(GaLayer(Layer(by_name["spread"], None), None))
    assert raw.any() and (~raw).any()
    assert modes[0] > 0 and modes[1] > 0
    raw, modes = _tile_modes(GaLayer(Layer(by_name["ragged-b6"], None), None))
    assert modes[0] > 0 and modes[1] > 0 and modes[2] > 0 and modes[3] == 0, modes


def test_ragged_lengths_and_every_tail(kvz, oracle):
    cfg = kvgen.KVConfig("lengths", 1, 20, 8, 2, 6, tail_min=1, tail_max=15, seed=41)
    lens = [0, 1, 15, 16, 17, 31, 32, 33, 47, 48, 50, 63, 64, 70, 80, 89, 95, 96, 97, 100]
    base = Layer(cfg, None, seq_lens=lens)
    ga = GaLayer(base, oracle)
    _check_codec(ga, "lengths")
    out = ga.run()
    out_r = base.run_raw()
    torch.cuda.synchronize()
    assert int(ga.status.item()) == 0
    ref, st = ga.oracle_attention(oracle)
    assert st == 0
    check_attention(out, ref, "lengths")
    assert torch.equal(out, out_r)
    assert not out[0].any()


def test_bad_entry_is_flagged_and_skipped(kvz, oracle):
    cfg = kvgen.KVConfig("bad-entry", 1, 3, 8, 2, 5, tail_min=2, tail_max=9, seed=51)
    base = Layer(cfg, None)
    ga = GaLayer(base, oracle)
    pid = int(base.full[1, 2])
    meta = ga.meta.clone()
    meta[pid, 1, 0] = -1  # KVZ_GA_ENTRY_INVALID
    o_meta = ga.o_meta.copy()
    o_meta[pid, 1, 0] = 0xFFFFFFFF
    st = kvz.new_status()
    out = ga.run(meta=meta, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & kvz.STATUS_BAD_META
    ref, ost = ga.oracle_attention(oracle, meta=o_meta)
    assert ost & 8
    check_attention(out, ref, "bad entry")


def test_arena_full_matches_oracle(kvz, oracle):
    """Cursor regions too small for every tile: the same tiles are missing on both sides."""
    cfg = kvgen.KVConfig("tight", 1, 2, 8, 2, 6, seed=52)
    base = Layer(cfg, None)
    ga = GaLayer(base, None)
    cur = np.array([[0, 47 * 9], [1000, 1000 + 47 * 30]], np.uint32)
    meta = torch.zeros_like(ga.meta)
    arena = torch.zeros_like(ga.arena)
    cursors = torch.from_numpy(cur.view(np.int32).copy()).cuda()
    st = kvz.new_status()
    s = base.src.cuda()
    kvz.ga_encode_pages(base.g_pool, ga.bases, s, s, base.dseq.cuda(), meta, arena, cursors, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvz.STATUS_ARENA_FULL
    o_meta = np.zeros((cfg.num_pages, cfg.hkv, 2), np.uint32)
    o_arena = np.zeros(ga.arena_bytes, np.uint8)
    o_cur = cur.copy()
    ost = oracle.ga_encode_pages(kvgen.bits(base.pool), ga.bases.cpu().numpy(), base.src.numpy(), base.src.numpy(),
                                 base.dseq.numpy(), o_meta, o_arena, o_cur, cfg.hkv)
    assert ost == 1
    assert np.array_equal(_np_meta(meta), o_meta)
    assert np.array_equal(arena.cpu().numpy(), o_arena)
    assert np.array_equal(cursors.cpu().numpy().view(np.uint32), o_cur)


def test_calibration_bad_page_and_empty_sample(kvz, oracle):
    cfg = kvgen.C0
    base = Layer(cfg, None)
    bases = torch.full((cfg.hkv, 2, 2, 128), 7, dtype=torch.uint8, device="cuda")
    st = kvz.new_status()
    kvz.ga_calibrate(base.g_pool, torch.zeros(0, dtype=torch.int32, device="cuda"), bases, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and not bases.any()  # no sample: all windows start at 0
    pages = torch.tensor([0, 3, 10_000, 5], dtype=torch.int32, device="cuda")
    kvz.ga_calibrate(base.g_pool, pages, bases, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvz.STATUS_BAD_INDEX
    ref = oracle.ga_calibrate_pool(kvgen.bits(base.pool), [0, 3, 5], cfg.hkv)
    assert np.array_equal(bases.cpu().numpy(), ref)
