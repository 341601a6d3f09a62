"""GPU codec parity: libkvz's encoder, placement scan and decoder against the CPU
oracle, bit for bit (ZipFusion "How it works" steps 1-4, metadata paragraph)."""
import numpy as np
import pytest
import torch

import kvgen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvz():
    from decode_attention_value_gb300 import _build

    _build.build()
    import decode_attention_value_gb300 as m

    return m


def encode_both(kvz, oracle, pool, src, dst, seq, n_meta, arena_bytes, cursors0):
    hkv = pool.shape[1]
    g_meta = torch.zeros((n_meta, hkv, 2), dtype=torch.int64, device="cuda")
    g_arena = torch.zeros(arena_bytes, dtype=torch.uint8, device="cuda")
    g_cur = torch.from_numpy(np.asarray(cursors0, np.uint32).view(np.int32).copy()).cuda()
    st = kvz.new_status()
    kvz.encode_pages(pool.cuda(), torch.as_tensor(src, dtype=torch.int32).cuda(),
                     torch.as_tensor(dst, dtype=torch.int32).cuda(), torch.as_tensor(seq, dtype=torch.int32).cuda(),
                     g_meta, g_arena, g_cur, st)
    torch.cuda.synchronize()
    o_meta = np.zeros((n_meta, hkv, 2), np.uint64)
    o_arena = np.zeros(arena_bytes, np.uint8)
    o_cur = np.asarray(cursors0, np.uint32).copy()
    o_st = oracle.encode_pages(kvgen.bits(pool), src, dst, seq, o_meta, o_arena, o_cur, hkv)
    gpu = (g_meta.cpu().numpy().view(np.uint64), g_arena.cpu().numpy(), g_cur.cpu().numpy().view(np.uint32),
           int(st.item()))
    return gpu, (o_meta, o_arena, o_cur, o_st)


def assert_same(gpu, ora):
    assert gpu[3] == ora[3], f"status {gpu[3]} vs oracle {ora[3]}"
    assert np.array_equal(gpu[2], ora[2]), "cursors differ"
    assert np.array_equal(gpu[0], ora[0]), "metadata differs"
    diff = np.nonzero(gpu[1] != ora[1])[0]
    assert diff.size == 0, f"arena differs at {diff[:8]} ({diff.size} bytes)"


def spread_cfg(lo, hi, seed, hkv=2):
    return kvgen.KVConfig(f"spread{lo}-{hi}", 1, 1, 4 * hkv, hkv, 8, spread=(lo, hi), seed=seed)


# KV head counts from 1 to 16
@pytest.mark.parametrize("cfg", [kvgen.C0, spread_cfg(8, 20, 5), spread_cfg(8, 14, 6), spread_cfg(16, 20, 7),
                                 kvgen.KVConfig("llama-like", 1, 1, 32, 8, 6, k_log2_sigma=(-4, 3),
                                                v_log2_sigma=(-3, 1), k_outlier_channels=4,
                                                k_outlier_scale=32.0, seed=9),
                                 spread_cfg(8, 20, 21, hkv=1), spread_cfg(8, 20, 22, hkv=3),
                                 kvgen.KVConfig("hkv16-two-pass", 1, 1, 32, 16, 9, k_log2_sigma=(-4, 3),
                                                v_log2_sigma=(-3, 1), k_outlier_channels=4,
                                                k_outlier_scale=32.0, seed=23)],
                         ids=lambda c: f"{c.name}-hkv{c.hkv}")
def test_encode_bit_exact(kvz, oracle, cfg):
    n = cfg.num_pages
    pool = kvgen.gen_pages(cfg, n)
    src = np.random.default_rng(cfg.seed).permutation(n).astype(np.int32)
    dst = np.arange(n, dtype=np.int32)
    seq = np.zeros(n, np.int32)
    gpu, ora = encode_both(kvz, oracle, pool, src, dst, seq, n, n * cfg.hkv * 8192 + 4096, [[3, 1 << 30]])
    assert_same(gpu, ora)


def test_encode_extremes_all_eligible_and_all_raw(kvz, oracle):
    # spread 8 -> every block eligible; spread 20 -> every block raw
    for lo_hi, expect_raw in (((8, 8), False), ((20, 20), True)):
        cfg = spread_cfg(*lo_hi, seed=11, hkv=4)
        pool = kvgen.gen_pages(cfg, cfg.num_pages)
        n = cfg.num_pages
        gpu, ora = encode_both(kvz, oracle, pool, np.arange(n, dtype=np.int32), np.arange(n, dtype=np.int32),
                               np.zeros(n, np.int32), n, n * 4 * 8192, [[0, 1 << 30]])
        assert_same(gpu, ora)
        tags = ora[0] >> np.uint64(32)
        all_raw = np.all(tags == np.uint64(0xFFFFFFFF))
        assert bool(all_raw) == expect_raw
        per_group = 16 if expect_raw else 12
        assert int(ora[2][0, 0]) == n * 4 * 2 * per_group


@pytest.mark.parametrize("hkv", [8, 16], ids=lambda h: f"hkv{h}")
def test_encode_many_cursors_and_scan_tiles(kvz, oracle, hkv):
    """Thousands of (page, head) pairs in ten cursors of 1 to 210 pages: segments that cross
    the placement scan's tiles."""
    cfg = kvgen.KVConfig("scan", 1, 1, 2 * hkv, hkv, 1200, k_log2_sigma=(-4, 3), v_log2_sigma=(-3, 1),
                         block_outlier_frac=0.2, seed=13)
    n = cfg.num_pages
    pool = kvgen.gen_pages(cfg, n)
    rng = np.random.default_rng(2)
    sizes = np.array([100, 150, 7, 149, 1, 133, 150, 150, 150, 210], np.int64)  # 10 cursors, 1200 pages
    assert sizes.sum() == n
    seq = np.repeat(np.arange(10, dtype=np.int32), sizes)
    worst = sizes * cfg.hkv * 2 * 16
    starts = np.concatenate([[5], 5 + np.cumsum(worst + 3)[:-1]])
    cursors = np.stack([starts, starts + worst], 1).astype(np.uint32)
    src = rng.permutation(n).astype(np.int32)
    dst = rng.permutation(n).astype(np.int32)
    arena_bytes = int(cursors[-1, 1]) * 256
    gpu, ora = encode_both(kvz, oracle, pool, src, dst, seq, n, arena_bytes, cursors)
    assert_same(gpu, ora)


def test_encode_error_paths_match_oracle(kvz, oracle):
    cfg = kvgen.C0
    n = 6
    pool = kvgen.gen_pages(cfg, n)
    ar = n * cfg.hkv * 8192
    # cursor region too small: later groups are marked invalid, nothing written past the end
    gpu, ora = encode_both(kvz, oracle, pool, np.arange(n, dtype=np.int32), np.arange(n, dtype=np.int32),
                           np.zeros(n, np.int32), n, ar, [[0, 100]])
    assert ora[3] == oracle.ARENA_FULL
    assert_same(gpu, ora)
    # arena smaller than the cursor claims
    gpu, ora = encode_both(kvz, oracle, pool, np.arange(n, dtype=np.int32), np.arange(n, dtype=np.int32),
                           np.zeros(n, np.int32), n, 90 * 256, [[0, 1 << 20]])
    assert ora[3] == oracle.ARENA_FULL
    assert_same(gpu, ora)
    # decreasing cursor order: nothing happens
    gpu, ora = encode_both(kvz, oracle, pool, np.arange(n, dtype=np.int32), np.arange(n, dtype=np.int32),
                           np.array([0, 0, 1, 1, 0, 1], np.int32), n, ar, [[0, 4000], [4000, 8000]])
    assert ora[3] == oracle.BAD_ORDER
    assert_same(gpu, ora)
    assert not gpu[0].any() and not gpu[1].any()
    # index out of range: nothing happens
    gpu, ora = encode_both(kvz, oracle, pool, np.array([0, 1, 2, 3, 4, 99], np.int32),
                           np.arange(n, dtype=np.int32), np.zeros(n, np.int32), n, ar, [[0, 4000]])
    assert ora[3] == oracle.BAD_INDEX
    assert_same(gpu, ora)


@pytest.mark.parametrize("cfg", [kvgen.C0, spread_cfg(8, 20, 17, hkv=8)], ids=lambda c: c.name)
def test_decode_bit_exact_and_bad_metadata(kvz, oracle, cfg):
    n = cfg.num_pages
    pool = kvgen.gen_pages(cfg, n)
    src = np.arange(n, dtype=np.int32)
    gpu, ora = encode_both(kvz, oracle, pool, src, src, np.zeros(n, np.int32), n, n * cfg.hkv * 8192, [[0, 1 << 30]])
    assert_same(gpu, ora)
    meta = torch.from_numpy(gpu[0].view(np.int64).copy()).cuda()
    arena = torch.from_numpy(gpu[1]).cuda()
    order = torch.from_numpy(np.random.default_rng(1).permutation(n).astype(np.int32)).cuda()
    out = torch.full((n, cfg.hkv, 2, 16, 128), 7, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    st = kvz.new_status()
    kvz.decode_blocks(meta, arena, order, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out.cpu().view(torch.int16), pool[order.cpu().long()].view(torch.int16))
    # corrupt metadata: bad tag byte, invalid offset, offset past the arena, page id out of range
    bad = gpu[0].copy()
    bad[0, 0, 1] = (bad[0, 0, 1] & np.uint64(0x00FFFFFFFFFFFFFF)) | np.uint64(0x9A << 56)
    bad[1, cfg.hkv - 1, 0] = np.uint64(0xFFFFFFFF) | (bad[1, cfg.hkv - 1, 0] & np.uint64(0xFFFFFFFF00000000))
    bad[2, 0, 0] = np.uint64(arena.numel() // 256 - 5) | (bad[2, 0, 0] & np.uint64(0xFFFFFFFF00000000))
    pages = np.array([0, 1, 2, 3, n + 4], np.int32)
    o_out, o_st = oracle.decode_pages(bad, gpu[1], pages, cfg.hkv)
    st.zero_()
    out = torch.empty((5, cfg.hkv, 2, 16, 128), dtype=torch.bfloat16, device="cuda")
    kvz.decode_blocks(torch.from_numpy(bad.view(np.int64).copy()).cuda(), arena, torch.from_numpy(pages).cuda(),
                      out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == o_st == (oracle.BAD_META | oracle.BAD_INDEX)
    assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), o_out)


@pytest.mark.parametrize("cfg", [kvgen.C0, spread_cfg(8, 20, 11, hkv=8),
                                 kvgen.KVConfig("llama-like-sizes", 1, 1, 32, 8, 40, k_log2_sigma=(-4, 3),
                                                v_log2_sigma=(-3, 1), k_outlier_channels=4,
                                                k_outlier_scale=32.0, seed=12)],
                         ids=lambda c: c.name)
def test_encode_sizes_match_the_oracle_placement(kvz, oracle, cfg):
    """kvz_encode_sizes (the size pass alone, for exact reservations): per page the
    granules of all its groups, each 3 or 4 per block by the oracle's own tags, and the
    distance the oracle's cursor moves over that page; a call with an out-of-range page id
    reads no page, reports 0 for every page and is flagged."""
    n = cfg.num_pages
    pool = kvgen.gen_pages(cfg, n)
    src = np.random.default_rng(cfg.seed + 1).permutation(n).astype(np.int32)
    g_sizes = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    st = kvz.new_status()
    kvz.encode_sizes(pool.cuda(), torch.from_numpy(src).cuda(), g_sizes, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = g_sizes.cpu().numpy().astype(np.int64)
    # oracle: encode the same pages one cursor per page, read sizes off the tags and cursors
    o_meta = np.zeros((n, cfg.hkv, 2), np.uint64)
    o_arena = np.zeros(n * cfg.hkv * 8192, np.uint8)
    per = cfg.hkv * 2 * 16
    cur = np.array([[i * per, (i + 1) * per] for i in range(n)], np.uint32)
    start = cur[:, 0].copy()
    assert oracle.encode_pages(kvgen.bits(pool), src, np.arange(n, dtype=np.int32), np.arange(n, dtype=np.int32),
                               o_meta, o_arena, cur, cfg.hkv) == 0
    tags = (o_meta >> np.uint64(32)).astype(np.uint64)
    raw = sum(((tags >> np.uint64(8 * j)) & np.uint64(0xFF)) == 0xFF for j in range(4)).sum(axis=(1, 2))
    from_tags = 3 * 4 * 2 * cfg.hkv + raw.astype(np.int64)
    assert np.array_equal(from_tags, cur[:, 0].astype(np.int64) - start)
    assert np.array_equal(got, from_tags)
    # an out-of-range page id: no sizes, BAD_INDEX
    bad = src.copy()
    bad[n // 2] = n + 5
    g_sizes.fill_(-1)
    st = kvz.new_status()
    kvz.encode_sizes(pool.cuda(), torch.from_numpy(bad).cuda(), g_sizes, st)
    torch.cuda.synchronize()
    assert int(st.item()) == kvz.STATUS_BAD_INDEX
    assert (g_sizes.cpu() == 0).all()


def _large_case(hkv, n, seed, cursors=10):
    """A pool of n pages (70-110 MB of BF16), placed through `cursors` cursors of ragged run
    lengths, shuffled sources and destinations."""
    cfg = kvgen.KVConfig("large", 1, 1, 2 * hkv, hkv, n, k_log2_sigma=(-4, 3), v_log2_sigma=(-3, 1),
                         block_outlier_frac=0.2, seed=seed)
    pool = kvgen.gen_pages(cfg, n)
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, n), cursors - 1, replace=False))
    sizes = np.diff(np.concatenate([[0], cuts, [n]]))
    seq = np.repeat(np.arange(cursors, dtype=np.int32), sizes)
    worst = sizes.astype(np.int64) * hkv * 2 * 16
    starts = np.concatenate([[7], 7 + np.cumsum(worst + 5)[:-1]])
    cur = np.stack([starts, starts + worst], 1).astype(np.uint32)
    return pool, rng.permutation(n).astype(np.int32), rng.permutation(n).astype(np.int32), seq, cur


@pytest.mark.parametrize("hkv,n", [(1, 9000), (2, 5000), (8, 1700)], ids=lambda v: str(v))
def test_encode_large_inputs(kvz, oracle, hkv, n):
    """Inputs larger than L2 through ragged cursors: bytes, metadata and cursors against
    the oracle."""
    pool, src, dst, seq, cur = _large_case(hkv, n, seed=50 + hkv)
    gpu, ora = encode_both(kvz, oracle, pool, src, dst, seq, n, int(cur[-1, 1]) * 256, cur)
    assert_same(gpu, ora)


def test_encode_large_arena_full_and_bad_index(kvz, oracle):
    hkv, n = 8, 1500
    pool, src, dst, seq, cur = _large_case(hkv, n, seed=61)
    # the fourth cursor's region holds a third of its worst case: some of its groups, in
    # the middle of the input, do not fit
    cur = cur.copy()
    cur[3, 1] = cur[3, 0] + (cur[3, 1] - cur[3, 0]) // 3
    gpu, ora = encode_both(kvz, oracle, pool, src, dst, seq, n, int(cur[-1, 1]) * 256, cur)
    assert ora[3] == oracle.ARENA_FULL
    assert_same(gpu, ora)
    # a source page out of range: nothing is written, cursors unchanged
    bad = src.copy()
    bad[n // 2] = n + 3
    gpu, ora = encode_both(kvz, oracle, pool, bad, dst, seq, n, int(cur[-1, 1]) * 256, cur)
    assert ora[3] == oracle.BAD_INDEX
    assert_same(gpu, ora)


def test_encode_reused_workspace_and_graph(kvz, oracle):
    """Two calls through one workspace, then the same call captured in a CUDA graph and
    replayed: the per-call state in the workspace (validation word, page-size sums) is
    reset by every call."""
    hkv, n = 4, 2400
    pool, src, dst, seq, cur = _large_case(hkv, n, seed=71)
    arena_bytes = int(cur[-1, 1]) * 256
    o_meta = np.zeros((n, hkv, 2), np.uint64)
    o_arena = np.zeros(arena_bytes, np.uint8)
    o_cur = cur.copy()
    assert oracle.encode_pages(kvgen.bits(pool), src, dst, seq, o_meta, o_arena, o_cur, hkv) == 0
    g_pool = pool.cuda()
    g_src, g_dst, g_seq = (torch.from_numpy(a).cuda() for a in (src, dst, seq))
    ws = torch.empty(kvz.encode_workspace_size(hkv, n), dtype=torch.uint8, device="cuda")
    meta = torch.zeros((n, hkv, 2), dtype=torch.int64, device="cuda")
    arena = torch.zeros(arena_bytes, dtype=torch.uint8, device="cuda")
    cursors = torch.zeros((len(cur), 2), dtype=torch.int32, device="cuda")
    st = kvz.new_status()
    cur0 = torch.from_numpy(cur.view(np.int32).copy()).cuda()

    def call():
        cursors.copy_(cur0)
        meta.zero_()
        arena.zero_()
        kvz.encode_pages(g_pool, g_src, g_dst, g_seq, meta, arena, cursors, st, workspace=ws)

    def check(what):
        torch.cuda.synchronize()
        assert int(st.item()) == 0, what
        assert np.array_equal(cursors.cpu().numpy().view(np.uint32), o_cur), what
        assert np.array_equal(meta.cpu().numpy().view(np.uint64), o_meta), what
        assert np.array_equal(arena.cpu().numpy(), o_arena), what

    for k in range(2):
        call()
        check(f"eager call {k}")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    check("side-stream call")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for k in range(2):
        g.replay()
        check(f"graph replay {k}")
