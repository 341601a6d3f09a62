"""GPU parity of the FP8 pages (GAAC "Relation to FP8 KV" with the group-adaptive codec):
the BF16 -> FP8 conversion over every BF16 word, bases, tile bytes, entries and cursors
bit-exact against the CPU oracle, bit-exact decode, and attention within the tolerance of
the fp64 oracle and bit-identical to the raw BF16 kernel over the same (FP8) values."""
import numpy as np
import pytest
import torch

import kvgen
from helpers import F8Layer, Layer, check_attention

pytestmark = pytest.mark.gpu

FMTS = [1, 2]  # E4M3, E5M2

CASES = [
    kvgen.C0,
    kvgen.C0_TAIL,
    kvgen.KVConfig("ragged-b6", 1, 6, 16, 4, 9, tail_min=1, tail_max=15, k_log2_sigma=(-4, 3),
                   v_log2_sigma=(-3, 1), k_outlier_channels=4, k_outlier_scale=32.0, block_outlier_frac=0.05,
                   block_outlier_log2=14, seed=31),
    kvgen.KVConfig("gqa1", 1, 3, 4, 4, 7, tail_min=3, tail_max=9, seed=32),
    kvgen.KVConfig("gqa8", 1, 5, 16, 2, 11, tail_min=1, tail_max=15, seed=36),
    kvgen.KVConfig("spread", 1, 2, 32, 8, 12, tail_min=1, tail_max=15, spread=(6, 12), seed=34),
    kvgen.KVConfig("gqa3", 1, 3, 6, 2, 7, tail_min=1, tail_max=15, k_log2_sigma=(-4, 3), seed=38),
    kvgen.KVConfig("gqa6", 1, 3, 12, 2, 9, tail_min=1, tail_max=15, v_log2_sigma=(-3, 1), seed=40),
    kvgen.KVConfig("llama-b4", 1, 4, 32, 8, 20, tail_min=1, tail_max=15, k_log2_sigma=(-4, 3),
                   v_log2_sigma=(-3, 1), k_outlier_channels=4, k_outlier_scale=32.0, seed=35),
]


def _u32(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("fmt", FMTS)
def test_conversion_of_every_bf16_word(oracle, fmt):
    """All 65,536 BF16 words as one pool (16 pages, 1 KV head), encoded and decoded."""
    import decode_attention_value_gb300 as kvz

    words = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(16, 1, 2, 16, 128)
    pool = torch.from_numpy(words.view(np.int16).copy()).cuda().view(torch.bfloat16)
    src = torch.arange(16, dtype=torch.int32, device="cuda")
    bases = torch.zeros((1, 2, 2, 128), dtype=torch.uint8, device="cuda")
    st = kvz.new_status()
    kvz.f8_calibrate(fmt, pool, src, bases, st)
    meta = torch.zeros((16, 1, 2), dtype=torch.int32, device="cuda")
    arena = torch.zeros(16 * 2 * 2048, dtype=torch.uint8, device="cuda")
    cur = torch.tensor([[0, 16 * 2 * 32]], dtype=torch.int32, device="cuda")
    kvz.f8_encode_pages(fmt, pool, bases, src, src, torch.zeros(16, dtype=torch.int32, device="cuda"), meta, arena,
                        cur, st)
    out = torch.empty((16, 1, 2, 16, 128), dtype=torch.uint8, device="cuda")
    kvz.f8_decode_blocks(fmt, meta, arena, bases, src, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want = oracle.f8_quantize(fmt, words)
    got = out.cpu().numpy()
    bad = np.flatnonzero(got.reshape(-1) != want.reshape(-1))
    assert bad.size == 0, [(hex(int(words.reshape(-1)[i])), hex(int(got.reshape(-1)[i])),
                            hex(int(want.reshape(-1)[i]))) for i in bad[:8]]
    # the oracle places the same tiles (same bases)
    o_meta = np.zeros((16, 1, 2), np.uint32)
    o_arena = np.zeros(arena.numel(), np.uint8)
    o_cur = np.array([[0, 16 * 2 * 32]], np.uint32)
    assert oracle.f8_encode_pages(fmt, words, bases.cpu().numpy(), np.arange(16, dtype=np.int32),
                                  np.arange(16, dtype=np.int32), np.zeros(16, np.int32), o_meta, o_arena, o_cur,
                                  1) == 0
    assert np.array_equal(_u32(meta), o_meta) and np.array_equal(arena.cpu().numpy(), o_arena)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_codec_and_attention(kvz_lib, oracle, fmt, cfg):
    kvz = kvz_lib
    base = Layer(cfg, None)
    f8 = F8Layer(base, fmt, oracle)
    assert np.array_equal(f8.bases.cpu().numpy(), f8.o_bases), "bases"
    assert np.array_equal(_u32(f8.meta), f8.o_meta), "entries"
    assert np.array_equal(f8.arena.cpu().numpy(), f8.o_arena), "tile bytes"
    assert np.array_equal(_u32(f8.cursors), f8.o_cursors), "cursors"
    if base.src.numel():
        out = torch.empty((base.src.numel(), cfg.hkv, 2, 16, 128), dtype=torch.uint8, device="cuda")
        st = kvz.new_status()
        kvz.f8_decode_blocks(fmt, f8.meta, f8.arena, f8.bases, base.src.cuda(), out, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert np.array_equal(out.cpu().numpy(), oracle.f8_quantize(fmt, kvgen.bits(base.pool)[base.src.numpy()]))
    got = f8.run()
    torch.cuda.synchronize()
    assert int(f8.status.item()) == 0
    ref, st = f8.oracle_attention(oracle)
    assert st == 0
    check_attention(got, ref, f"{cfg.name} fp8 {fmt}")
    # the raw BF16 kernel over a pool whose completed pages hold the same FP8 values
    pool = kvgen.bits(base.pool).copy()
    src = base.src.numpy()
    if src.size:
        q8 = oracle.f8_quantize(fmt, pool[src])
        vals = np.vectorize(lambda b: oracle.f8_value(fmt, b), otypes=[np.float32])(q8)
        pool[src] = (vals.view(np.uint32) >> 16).astype(np.uint16)
    g_pool = torch.from_numpy(pool.view(np.int16)).cuda().view(torch.bfloat16)
    out_r = torch.empty_like(got)
    st = kvz.new_status()
    kvz.decode_attention_raw(base.g_q, base.raw_table().cuda(), base.seq_lens.cuda(), g_pool, out_r, st,
                             workspace=base.workspace(True))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # FP8 pages are multiplied in f16, the raw kernel's pages in BF16: the K and V values
    # are the same, and so are the queries (exact in f16 here); P = hi + lo keeps ~22 bits
    # in f16 against ~16 in BF16, so the outputs agree to ~1e-5 of their scale
    scale = float(out_r.float().pow(2).mean().sqrt())
    assert float((got - out_r).abs().max()) <= 2e-4 * max(scale, 1e-30)


@pytest.fixture(scope="module")
def kvz_lib():
    from decode_attention_value_gb300 import _build

    _build.build()
    import decode_attention_value_gb300 as m

    return m


@pytest.mark.parametrize("fmt", FMTS)
def test_bad_entry_flagged(kvz_lib, oracle, fmt):
    kvz = kvz_lib
    cfg = kvgen.KVConfig("bad-entry", 1, 3, 8, 2, 5, tail_min=2, tail_max=9, seed=51)
    base = Layer(cfg, None)
    f8 = F8Layer(base, fmt, oracle)
    pid = int(base.full[1, 2])
    meta = f8.meta.clone()
    meta[pid, 0, 1] = -1
    o_meta = f8.o_meta.copy()
    o_meta[pid, 0, 1] = 0xFFFFFFFF
    st = kvz.new_status()
    out = f8.run(meta=meta, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & kvz.STATUS_BAD_META
    ref, ost = f8.oracle_attention(oracle, meta=o_meta)
    assert ost & 8
    check_attention(out, ref, "bad entry")


@pytest.mark.parametrize("fmt", [1, 2], ids=["e4m3", "e5m2"])
def test_query_beyond_f16_range_is_flagged(kvz_lib, oracle, fmt):
    """FP8 pages are multiplied in f16: a finite BF16 query element beyond the f16 range
    sets KVZ_STATUS_Q_RANGE (queries inside the range leave the status clear)."""
    kvz = kvz_lib
    cfg = kvgen.KVConfig("q-range", 1, 2, 8, 2, 4, tail_min=1, tail_max=9, seed=61)
    base = Layer(cfg, None)
    f8 = F8Layer(base, fmt, oracle)
    st = kvz.new_status()
    f8.run(status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    base.g_q[1, 5, 17] = 1.0e5  # BF16 99840: finite, above 65504
    st = kvz.new_status()
    f8.run(status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvz.STATUS_Q_RANGE


def test_e4m3_ignores_b4_entries(kvz_lib, oracle):
    """E4M3 takes b4 = 0 whatever the bases table holds: with junk b4 entries the encoder
    writes the same tiles (and the oracle agrees), and decode and attention read them the
    same way."""
    kvz = kvz_lib
    cfg = kvgen.KVConfig("e4-junk-b4", 1, 3, 8, 2, 9, tail_min=1, tail_max=15, k_log2_sigma=(-4, 3),
                         v_log2_sigma=(-3, 1), k_outlier_channels=4, k_outlier_scale=32.0, seed=63)
    base = Layer(cfg, None)
    f8 = F8Layer(base, 1, oracle)
    assert np.array_equal(f8.arena.cpu().numpy(), f8.o_arena)
    junk = f8.bases.clone()
    g = torch.Generator().manual_seed(5)
    junk[:, :, 1, :] = torch.randint(1, 256, junk[:, :, 1, :].shape, generator=g, dtype=torch.uint8).cuda()
    meta = torch.zeros_like(f8.meta)
    arena = torch.zeros_like(f8.arena)
    cur = torch.from_numpy(f8.cursors0.view(np.int32).copy()).cuda()
    st = kvz.new_status()
    s = base.src.cuda()
    kvz.f8_encode_pages(1, base.g_pool, junk, s, s, base.dseq.cuda(), meta, arena, cur, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(meta, f8.meta) and torch.equal(arena, f8.arena)
    o_meta = np.zeros_like(f8.o_meta)
    o_arena = np.zeros_like(f8.o_arena)
    o_cur = f8.cursors0.copy()
    src = base.src.numpy()
    assert oracle.f8_encode_pages(1, f8.o_pool, junk.cpu().numpy(), src, src, base.dseq.numpy(), o_meta, o_arena,
                                  o_cur, cfg.hkv) == 0
    assert np.array_equal(o_arena, f8.o_arena) and np.array_equal(o_meta, f8.o_meta)
    out = torch.empty((s.numel(), cfg.hkv, 2, 16, 128), dtype=torch.uint8, device="cuda")
    kvz.f8_decode_blocks(1, meta, arena, junk, s, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(out.cpu().numpy(), oracle.f8_quantize(1, kvgen.bits(base.pool)[src]))
    want = f8.run()
    got = torch.empty_like(want)
    kvz.f8_decode_attention(1, base.g_q, base.full.cuda(), base.seq_lens.cuda(), base.tail.cuda(), meta, arena,
                            junk, base.g_pool, got, st, workspace=base.workspace(False))
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and torch.equal(got, want)
