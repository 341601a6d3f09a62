"""GPU decode-attention parity (GAAC "Attention with On-the-Fly Decompression";
ZipFusion "How it works"): the compressed and raw kernels against the fp64 CPU oracle
within the stated tolerance, and against each other bit for bit."""
import numpy as np
import pytest
import torch

import kvgen
from helpers import Layer, check_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvz():
    from decode_attention_value_gb300 import _build

    _build.build()
    import decode_attention_value_gb300 as m

    return m


def run_and_check(layer, oracle, what):
    out_c = layer.run_compressed()
    out_r = layer.run_raw()
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0, f"{what}: status {int(layer.status.item())}"
    ref, st = layer.oracle_attention(oracle)
    assert st == 0
    check_attention(out_c, ref, what + " compressed")
    check_attention(out_r, ref, what + " raw")
    assert torch.equal(out_c, out_r), f"{what}: compressed and raw outputs differ"
    return out_c, ref


CASES = [
    kvgen.C0,
    kvgen.C0_TAIL,
    kvgen.KVConfig("ragged-b6", 1, 6, 16, 4, 9, tail_min=1, tail_max=15, k_log2_sigma=(-4, 3),
                   v_log2_sigma=(-3, 1), k_outlier_channels=4, k_outlier_scale=32.0, block_outlier_frac=0.05,
                   block_outlier_log2=14, seed=31),
    kvgen.KVConfig("gqa1", 1, 3, 4, 4, 7, tail_min=3, tail_max=9, seed=32),
    kvgen.KVConfig("gqa2", 1, 3, 8, 4, 7, tail_min=3, tail_max=9, seed=33),
    # G = 8 (e.g. 64 query heads over 8 KV heads): every MMA column a head
    kvgen.KVConfig("gqa8", 1, 5, 16, 2, 11, tail_min=1, tail_max=15, k_log2_sigma=(-4, 3), v_log2_sigma=(-3, 1),
                   k_outlier_channels=4, k_outlier_scale=32.0, block_outlier_frac=0.05, seed=36),
    kvgen.KVConfig("gqa8-llama70b-shape", 1, 4, 64, 8, 40, tail_min=1, tail_max=15, k_log2_sigma=(-4, 3),
                   v_log2_sigma=(-3, 1), k_outlier_channels=4, k_outlier_scale=32.0, seed=37),
    kvgen.KVConfig("spread", 1, 2, 32, 8, 12, tail_min=1, tail_max=15, spread=(8, 20), seed=34),
    # group sizes that are not powers of two: G = 3 takes the spare-column kernel with one
    # zero head column, G = 5, 6, 7 the all-heads kernel with zero columns
    kvgen.KVConfig("gqa3", 1, 3, 6, 2, 7, tail_min=1, tail_max=15, k_log2_sigma=(-4, 3), seed=38),
    kvgen.KVConfig("gqa5", 1, 2, 20, 4, 6, tail_min=2, tail_max=13, seed=39),
    kvgen.KVConfig("gqa6", 1, 3, 12, 2, 9, tail_min=1, tail_max=15, v_log2_sigma=(-3, 1), seed=40),
    kvgen.KVConfig("gqa7", 1, 2, 14, 2, 5, tail_min=3, tail_max=9, seed=43),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_attention_matches_oracle(kvz, oracle, cfg):
    run_and_check(Layer(cfg, oracle), oracle, cfg.name)


def test_ragged_lengths_and_every_tail(kvz, oracle):
    """Lengths 0..(pages*16): empty, tail-only, every tail length 0..15, full pages."""
    cfg = kvgen.KVConfig("lengths", 1, 20, 8, 2, 6, tail_min=1, tail_max=15, seed=41)
    lens = [0, 1, 15, 16, 17, 31, 32, 33, 47, 48, 50, 63, 64, 70, 80, 89, 95, 96, 97, 100]
    layer = Layer(cfg, oracle, seq_lens=lens)
    out, ref = run_and_check(layer, oracle, "lengths")
    assert not out[0].any()  # empty context -> zero output


def test_many_splits_long_context(kvz, oracle):
    """Few long sequences: every (sequence, head) unit is cut across many CTAs."""
    cfg = kvgen.KVConfig("long", 1, 2, 8, 2, 300, tail_min=5, tail_max=11, k_log2_sigma=(-4, 3),
                         v_log2_sigma=(-3, 1), seed=42)
    run_and_check(Layer(cfg, oracle), oracle, "long")


def test_bad_metadata_page_is_skipped(kvz, oracle):
    cfg = kvgen.C0_TAIL
    layer = Layer(cfg, oracle)
    bad_o = layer.o_meta.copy()
    victim = int(layer.full[0, 3])
    bad_o[victim, 1, 1] = np.uint64(0xFFFFFFFF) | (bad_o[victim, 1, 1] & np.uint64(0xFFFFFFFF00000000))
    bad_g = layer.meta.clone()
    bad_g[victim, 1, 1] = torch.from_numpy(bad_o[victim, 1, 1:2].view(np.int64)).cuda()
    st = kvz.new_status()
    out = layer.run_compressed(meta=bad_g, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvz.STATUS_BAD_META
    ref, o_st = layer.oracle_attention(oracle, meta=bad_o)
    assert o_st == oracle.BAD_META
    check_attention(out, ref, "bad meta")


def test_missing_tail_page_is_flagged(kvz, oracle):
    cfg = kvgen.C0_TAIL
    layer = Layer(cfg, oracle)
    layer.tail = torch.full_like(layer.tail, -1)
    st = kvz.new_status()
    layer.run_compressed(status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & kvz.STATUS_BAD_TAIL


def test_full_size_layer_all_outputs(kvz, oracle):
    """The Llama-3.1-8B-shaped layer (batch 32, 32/8 heads, 2048 + tail tokens, shuffled
    pages) in the bench's launch configuration: every output against the fp64 oracle
    run over the oracle's own encoding of every page."""
    layer = Layer(kvgen.C1, oracle)
    out_c = layer.run_compressed()
    out_r = layer.run_raw()
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    assert torch.equal(out_c, out_r)
    ref, st = layer.oracle_attention(oracle, nthreads=16)
    assert st == 0
    check_attention(out_c, ref, "C1 layer")


def _decompress_first(kvz, layer):
    """Decompress-first composition: kvz_decode_blocks of every compressed page into a
    BF16 scratch pool (in table order), each sequence's raw tail page copied beside them,
    then kvz_decode_attention_raw over the scratch pool with a table one column wider
    than the compressed call's (the same work split)."""
    cfg = layer.cfg
    B, nf = cfg.batch, cfg.full_pages
    full = layer.full.cuda()
    scratch = torch.empty((B * nf + B, cfg.hkv, 2, 16, 128), dtype=torch.bfloat16, device="cuda")
    st = kvz.new_status()
    n_full = (layer.seq_lens // 16).tolist()
    ids = torch.arange(B * nf, dtype=torch.int32).view(B, nf)
    for b in range(B):  # only the completed pages are encoded; the rest of each row stays unused
        if n_full[b]:
            kvz.decode_blocks(layer.meta, layer.arena, full[b, : n_full[b]].contiguous(),
                              scratch[b * nf: b * nf + n_full[b]], st)
    tails = layer.tail.clamp_min(0).long().cuda()
    scratch[B * nf:] = layer.g_pool[tails]
    # row b: its decoded pages, then its tail at column n_full[b] (unused when the length is
    # a whole number of pages); columns past the sequence's pages are never read
    table = torch.full((B, nf + 1), -1, dtype=torch.int32)
    for b in range(B):
        table[b, : n_full[b]] = ids[b, : n_full[b]]
        table[b, n_full[b]] = B * nf + b
    out = torch.empty((B, cfg.hq, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(kvz.attention_workspace_size(cfg.hkv, B, cfg.hq, nf + 1), dtype=torch.uint8, device="cuda")
    kvz.decode_attention_raw(layer.g_q, table.contiguous().cuda(), layer.seq_lens.cuda(), scratch, out, st,
                             workspace=ws)
    return out, st


@pytest.mark.parametrize("cfg", [kvgen.C0_TAIL, CASES[2], kvgen.KVConfig(
    "df-lengths", 1, 9, 8, 2, 6, tail_min=1, tail_max=15, seed=44)], ids=lambda c: c.name)
def test_decompress_first_matches_oracle(kvz, oracle, cfg):
    """The decompress-first pipeline (standalone decode, then the raw kernel) gives the
    fp64 oracle's attention within the tolerance and the fused kernel's output bit for
    bit; with ragged lengths, including whole-page lengths with no tail."""
    lens = [0, 16, 17, 40, 64, 65, 90, 95, 96] if cfg.name == "df-lengths" else None
    layer = Layer(cfg, oracle, seq_lens=lens)
    out_df, st = _decompress_first(kvz, layer)
    out_c = layer.run_compressed()
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(layer.status.item()) == 0
    ref, ost = layer.oracle_attention(oracle)
    assert ost == 0
    check_attention(out_df, ref, cfg.name + " decompress-first")
    assert torch.equal(out_df, out_c), "decompress-first and fused outputs differ"


def test_largest_batch_and_beyond(kvz, oracle):
    """The largest batch the kernel takes (1024 sequences: its per-sequence tables in shared
    memory lower occupancy to fewer CTAs per SM), ragged lengths with empty sequences;
    one more sequence is refused on the host."""
    cfg = kvgen.KVConfig("max-batch", 1, 1024, 8, 2, 2, tail_min=1, tail_max=15, seed=61)
    rng = np.random.default_rng(61)
    lens = rng.integers(0, 2 * 16 + 16, 1024)
    lens[::97] = 0
    layer = Layer(cfg, oracle, seq_lens=lens.astype(np.int32))
    run_and_check(layer, oracle, "batch 1024")
    q = torch.zeros((1025, 8, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((1025, 8, 128), dtype=torch.float32, device="cuda")
    ids = torch.zeros((1025, 1), dtype=torch.int32, device="cuda")
    lens1 = torch.zeros(1025, dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvz.KvzError) as e:
        kvz.decode_attention_raw(q, ids, lens1, layer.g_pool, out, kvz.new_status(), workspace=ws)
    assert e.value.code == -2  # KVZ_ERR_UNSUPPORTED


def test_corrupt_metadata_fuzz(kvz, oracle):
    """Random unusable metadata words (invalid tag bytes, offsets past the arena, the
    unwritten-group marker) on random pages: every one is flagged, no page is read from
    outside the arena, and the output equals the oracle's with the same pages left out."""
    cfg = kvgen.KVConfig("fuzz", 1, 6, 16, 4, 8, tail_min=1, tail_max=15, seed=71)
    layer = Layer(cfg, oracle)
    rng = np.random.default_rng(71)
    meta = layer.meta.clone()
    o_meta = layer.o_meta.copy()
    pages = rng.choice(layer.src.numpy(), 10, replace=False)
    arena_granules = layer.arena_bytes // 256
    for k, p in enumerate(pages):
        h, kv = int(rng.integers(0, cfg.hkv)), int(rng.integers(0, 2))
        word = int(o_meta[p, h, kv])
        kind = k % 3
        if kind == 0:  # a tag byte between 0x80 and 0xFE
            j = int(rng.integers(0, 4))
            word = (word & ~(0xFF << (32 + 8 * j))) | (int(rng.integers(0x80, 0xFF)) << (32 + 8 * j))
        elif kind == 1:  # a group that would end past the arena
            word = (word & ~0xFFFFFFFF) | int(rng.integers(arena_granules - 8, 0xFFFFFFF0))
        else:  # the unwritten-group marker
            word = (word & ~0xFFFFFFFF) | 0xFFFFFFFF
        o_meta[p, h, kv] = np.uint64(word)
        meta[p, h, kv] = int(np.uint64(word).view(np.int64))
    st = kvz.new_status()
    out = layer.run_compressed(meta=meta, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvz.STATUS_BAD_META
    ref, ost = layer.oracle_attention(oracle, meta=o_meta)
    assert ost == 8
    check_attention(out, ref, "fuzzed metadata")


def test_concurrent_streams_and_host_threads(kvz, oracle):
    """Calls on two streams at once, each with its own workspace and output, and calls
    from two host threads: the library keeps no per-call state outside its arguments, so
    every output equals the one from sequential calls, bit for bit."""
    import threading

    cfgs = [kvgen.KVConfig("conc-a", 1, 12, 32, 8, 40, tail_min=1, tail_max=15, k_log2_sigma=(-4, 3),
                           v_log2_sigma=(-3, 1), seed=71),
            kvgen.KVConfig("conc-b", 1, 5, 16, 2, 90, tail_min=1, tail_max=15, spread=(8, 20), seed=72)]
    layers = [Layer(c, oracle) for c in cfgs]
    want = []
    for layer in layers:
        out_c, out_r = layer.run_compressed(), layer.run_raw()
        torch.cuda.synchronize()
        assert torch.equal(out_c, out_r)
        ref, st = layer.oracle_attention(oracle)
        assert st == 0
        check_attention(out_c, ref, layer.cfg.name)
        want.append(out_c.clone())

    # two streams, both layers and both kernels on each, several rounds
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    outs = []
    for rnd in range(3):
        for k, layer in enumerate(layers):
            s = streams[(k + rnd) % 2]
            with torch.cuda.stream(s):
                outs.append((k, layer.run_compressed(), layer.run_raw()))
    torch.cuda.synchronize()
    for k, out_c, out_r in outs:
        assert torch.equal(out_c, want[k]) and torch.equal(out_r, want[k]), cfgs[k].name

    # two host threads, each with its own stream
    errors, results = [], {}

    def worker(k):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                res = [layers[k].run_compressed() for _ in range(4)]
            s.synchronize()
            results[k] = res
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for k in range(2):
        assert all(torch.equal(o, want[k]) for o in results[k]), cfgs[k].name
    assert all(int(layer.status.item()) == 0 for layer in layers)
