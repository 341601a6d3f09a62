"""CPU checks of the C-ABI boundary: libkvz.so loads, exports every function that
include/kvz.h declares, rejects bad arguments on the host before any launch, and its
host-side chunk allocator (GAAC "Block-Wise Compression Scheduling"; ZipFusion memory
manager paragraph) keeps every encoded group inside its sequence's chunk when the
CPU oracle stands in for the device."""
import ctypes
import os
import re

import numpy as np
import pytest

import kvgen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvz():
    from decode_attention_value_gb300 import _build

    _build.build()
    import decode_attention_value_gb300 as m

    return m


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b(kvz_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_four_calls():
    names = declared_functions()
    for call in ("kvz_encode_pages", "kvz_decode_blocks", "kvz_decode_attention", "kvz_decode_attention_raw"):
        assert call in names


def test_library_exports_every_declared_symbol(kvz):
    lib = ctypes.CDLL(kvz._build.LIB)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(kvz.EXPORTS) <= set(declared_functions())


def test_strerror(kvz):
    lib = kvz.lib()
    assert lib.kvz_strerror(0) == b"ok"
    for code in range(-7, 0):
        assert lib.kvz_strerror(code) not in (b"", b"unknown error")


def _dims(kvz, hkv=8, d=128, p=16):
    return kvz.Dims(hkv, d, p)


def test_host_rejects_bad_arguments(kvz):
    lib = kvz.lib()
    E = dict(inval=-1, unsup=-2, align=-3, ws=-4)
    fake = 1 << 20  # never dereferenced: every call below returns before any launch
    # shapes other than head_dim 128 / page 16 are unsupported, Hkv < 1 is invalid
    assert lib.kvz_encode_pages(_dims(kvz, d=64), fake, 1, fake, fake, fake, 1, fake, 1, fake, 1 << 20, fake, 1,
                                fake, 1 << 20, fake, None) == E["unsup"]
    assert lib.kvz_encode_pages(_dims(kvz, hkv=0), fake, 1, fake, fake, fake, 1, fake, 1, fake, 1 << 20, fake, 1,
                                fake, 1 << 20, fake, None) == E["inval"]
    # n = 0 is a no-op, negative n invalid
    assert lib.kvz_encode_pages(_dims(kvz), None, 0, None, None, None, 0, None, 0, None, 0, None, 0, None, 0,
                                None, None) == 0
    assert lib.kvz_encode_pages(_dims(kvz), fake, 1, fake, fake, fake, -1, fake, 1, fake, 1 << 20, fake, 1,
                                fake, 1 << 20, fake, None) == E["inval"]
    # null pointer / misaligned arena / short workspace
    assert lib.kvz_encode_pages(_dims(kvz), fake, 1, None, fake, fake, 1, fake, 1, fake, 1 << 20, fake, 1,
                                fake, 1 << 20, fake, None) == E["inval"]
    assert lib.kvz_encode_pages(_dims(kvz), fake, 1, fake, fake, fake, 1, fake, 1, fake + 16, 1 << 20, fake, 1,
                                fake, 1 << 20, fake, None) == E["align"]
    ws = kvz.encode_workspace_size(8, 10)
    # per-(page, head) sizes and block tags, per-page sizes and positions
    assert ws >= 10 * 8 * (4 + 8) + 2 * 10 * 4
    for hkv, n in ((1, 1), (2, 7), (8, 4096)):  # grows with the call, stays 16-byte granular
        w = kvz.encode_workspace_size(hkv, n)
        assert w % 8 == 0 and w >= n * hkv * 12 + 2 * n * 4 + 16
    assert lib.kvz_encode_pages(_dims(kvz), fake, 10, fake, fake, fake, 10, fake, 10, fake, 1 << 20, fake, 1,
                                fake, ws - 1, fake, None) == E["ws"]
    # decode: misaligned output
    assert lib.kvz_decode_blocks(_dims(kvz), fake, 1, fake, 1 << 20, fake, 1, fake + 2, fake, None) == E["align"]
    assert lib.kvz_decode_blocks(_dims(kvz), None, 0, None, 0, None, 0, None, None, None) == 0
    # attention: the query heads must be a whole multiple (1 to 8) of the KV heads
    assert lib.kvz_decode_attention(_dims(kvz), 2, 12, fake, fake, 4, fake, fake, fake, 1, fake, 1 << 20, fake, 1,
                                    fake, fake, 1 << 20, fake, None) == E["inval"]
    assert lib.kvz_decode_attention(_dims(kvz), 2, 128, fake, fake, 4, fake, fake, fake, 1, fake, 1 << 20, fake, 1,
                                    fake, fake, 1 << 20, fake, None) == E["unsup"]
    assert lib.kvz_decode_attention_raw(_dims(kvz), 2, 32, fake + 8, fake, 4, fake, fake, 1, fake, fake, 1 << 20,
                                        fake, None) == E["align"]
    assert lib.kvz_decode_attention_raw(_dims(kvz), 0, 32, None, None, 0, None, None, 0, None, None, 0, None,
                                        None) == 0
    assert lib.kvz_apply_cursor_updates(None, None, None, 0, None, 0, None) == 0


def test_host_rejects_bad_tile_arguments(kvz):
    """The group-adaptive and FP8 tile calls check their arguments on the host as the
    12-bit calls do: shapes, formats, null pointers, alignment (64-byte arena, 4/8-byte
    entries, 16-byte bases for the encoders) and the encoder workspace, all before any
    launch (fake pointers are never dereferenced)."""
    lib = kvz.lib()
    E = dict(inval=-1, unsup=-2, align=-3, ws=-4)
    fake = 1 << 20
    d, d64, d0 = _dims(kvz), _dims(kvz, d=64), _dims(kvz, hkv=0)
    M = 1 << 20
    # ---- calibration: shapes, null bases, null sample, misaligned pool / sample ----
    assert lib.kvz_ga_calibrate(d64, fake, 1, fake, 1, fake, fake, None) == E["unsup"]
    assert lib.kvz_ga_calibrate(d0, fake, 1, fake, 1, fake, fake, None) == E["inval"]
    assert lib.kvz_ga_calibrate(d, fake, 1, fake, -1, fake, fake, None) == E["inval"]
    assert lib.kvz_ga_calibrate(d, fake, 1, fake, 1, None, fake, None) == E["inval"]
    assert lib.kvz_ga_calibrate(d, fake, 1, None, 1, fake, fake, None) == E["inval"]
    assert lib.kvz_ga_calibrate(d, fake + 8, 1, fake, 1, fake, fake, None) == E["align"]
    assert lib.kvz_ga_calibrate(d, fake, 1, fake + 2, 1, fake, fake, None) == E["align"]
    for fmt in (0, 3, -1):  # only KVZ_F8_E4M3 (1) and KVZ_F8_E5M2 (2) exist
        assert lib.kvz_f8_calibrate(d, fmt, fake, 1, fake, 1, fake, fake, None) == E["inval"]
    assert lib.kvz_f8_calibrate(d64, 1, fake, 1, fake, 1, fake, fake, None) == E["unsup"]
    assert lib.kvz_f8_calibrate(d, 2, fake, 1, fake, 1, None, fake, None) == E["inval"]
    assert lib.kvz_f8_calibrate(d, 1, fake + 8, 1, fake, 1, fake, fake, None) == E["align"]

    # ---- encoders: n = 0 no-op, bad n, nulls, alignment of every buffer, short workspace ----
    def ga_enc(dims=d, pool=fake, bases=fake, src=fake, n=10, meta=fake, arena=fake, cur=fake, ws=fake,
               ws_bytes=M, status=fake):
        return lib.kvz_ga_encode_pages(dims, pool, 64, bases, src, src, src, n, meta, 64, arena, M, cur, 4, ws,
                                       ws_bytes, status, None)

    def f8_enc(fmt=1, dims=d, pool=fake, bases=fake, src=fake, n=10, meta=fake, arena=fake, cur=fake, ws=fake,
               ws_bytes=M, status=fake):
        return lib.kvz_f8_encode_pages(dims, fmt, pool, 64, bases, src, src, src, n, meta, 64, arena, M, cur, 4,
                                       ws, ws_bytes, status, None)

    for enc in (ga_enc, f8_enc):
        assert enc(n=0, pool=None, bases=None, src=None, meta=None, arena=None, cur=None, ws=None,
                   status=None) == 0
        assert enc(dims=d64) == E["unsup"]
        assert enc(dims=d0) == E["inval"]
        assert enc(n=-1) == E["inval"]
        for k in ("pool", "bases", "src", "meta", "arena", "cur", "ws", "status"):
            assert enc(**{k: None}) == E["inval"], k
        assert enc(pool=fake + 8) == E["align"]
        assert enc(bases=fake + 8) == E["align"]   # bases: 16-byte aligned
        assert enc(meta=fake + 4) == E["align"]    # 4-byte entries read in K/V pairs: 8-byte aligned
        assert enc(arena=fake + 32) == E["align"]  # 64-byte granules
        assert enc(cur=fake + 4) == E["align"]
        assert enc(ws=fake + 8) == E["align"]
        assert enc(ws_bytes=kvz.encode_workspace_size(8, 10) - 1) == E["ws"]
    for fmt in (0, 3):
        assert f8_enc(fmt=fmt) == E["inval"]

    # ---- standalone decoders ----
    def ga_dec(meta=fake, arena=fake, bases=fake, page=fake, n=4, out=fake, status=fake):
        return lib.kvz_ga_decode_blocks(d, meta, 64, arena, M, bases, page, n, out, status, None)

    def f8_dec(fmt=2, meta=fake, arena=fake, bases=fake, page=fake, n=4, out=fake, status=fake):
        return lib.kvz_f8_decode_blocks(d, fmt, meta, 64, arena, M, bases, page, n, out, status, None)

    for dec in (ga_dec, f8_dec):
        assert dec(n=0, meta=None, arena=None, bases=None, page=None, out=None, status=None) == 0
        assert dec(n=-1) == E["inval"]
        for k in ("meta", "arena", "bases", "page", "out", "status"):
            assert dec(**{k: None}) == E["inval"], k
        assert dec(meta=fake + 2) == E["align"]
        assert dec(arena=fake + 32) == E["align"]
        assert dec(out=fake + 8) == E["align"]
    assert f8_dec(bases=fake + 1) == E["align"]
    assert f8_dec(fmt=0) == E["inval"]

    # ---- attention over tiles: GQA shape, nulls, alignment ----
    def ga_att(B=2, hq=32, q=fake, tail=fake, meta=fake, arena=fake, bases=fake, ws=fake):
        return lib.kvz_ga_decode_attention(d, B, hq, q, fake, 4, fake, tail, meta, 64, arena, M, bases, fake, 1,
                                           fake, ws, M, fake, None)

    def f8_att(fmt=1, B=2, hq=32, q=fake, tail=fake, meta=fake, arena=fake, bases=fake, ws=fake):
        return lib.kvz_f8_decode_attention(d, fmt, B, hq, q, fake, 4, fake, tail, meta, 64, arena, M, bases, fake,
                                           1, fake, ws, M, fake, None)

    for att in (ga_att, f8_att):
        assert att(B=0, q=None, tail=None, meta=None, arena=None, bases=None, ws=None) == 0
        assert att(hq=12) == E["inval"]   # not a whole multiple of the 8 KV heads
        assert att(hq=128) == E["unsup"]  # G = 16 > 8
        assert att(q=fake + 8) == E["align"]
        assert att(ws=fake + 8) == E["align"]
        for k in ("tail", "meta", "arena", "bases", "q", "ws"):
            assert att(**{k: None}) == E["inval"], k
        assert att(meta=fake + 4) == E["align"]
        assert att(arena=fake + 32) == E["align"]
        assert att(bases=fake + 1) == E["align"]
        assert att(tail=fake + 2) == E["align"]
    for fmt in (0, 3):
        assert f8_att(fmt=fmt) == E["inval"]


# --------------------------------------------------------------------------------------
# allocator
# --------------------------------------------------------------------------------------
def test_allocator_reserve_release_stats(kvz):
    hkv = 2
    chunk = 4 * 64  # granules: room for 4 worst-case pages (64 granules each at Hkv 2)
    a = kvz.Allocator(arena_bytes=chunk * 256 * 3, chunk_granules=chunk, num_cursors=4, num_kv_heads=hkv)
    assert a.stats()["chunks_free"] == 3
    t1, up = a.reserve([0, 1], [2, 1])
    assert up == [(0, 0, chunk), (1, chunk, 2 * chunk)]  # chunk 0 first, then chunk 1
    t2, up = a.reserve([0], [2])  # 2 + 2 worst-case pages still fit chunk 0
    assert up == []
    t3, up = a.reserve([0], [1])  # a fifth worst-case page does not
    assert up == [(0, 2 * chunk, 3 * chunk)]
    with pytest.raises(kvz.KvzError) as e:
        a.reserve([2], [1])  # no chunk left
    assert e.value.code == kvz.ERR_OUT_OF_SPACE
    with pytest.raises(kvz.KvzError):
        a.reserve([3], [5])  # more than a chunk in one call
    st = a.stats()
    assert st["chunks_held"] == 3 and st["chunks_free"] == 0
    a.release(1)
    assert a.stats()["chunks_free"] == 1
    t4, up = a.reserve([2], [1])
    assert up == [(2, chunk, 2 * chunk)]  # the released chunk is reused


def test_allocator_observe_tightens_bound(kvz):
    hkv = 1  # worst case per page: 2 groups x 16 granules = 32 granules
    chunk = 90
    a = kvz.Allocator(arena_bytes=chunk * 256 * 2, chunk_granules=chunk, num_cursors=1, num_kv_heads=hkv)
    t, up = a.reserve([0], [2])
    assert up == [(0, 0, chunk)]
    assert a.stats()["used_bytes_bound"] == 64 * 256
    # the device used 2 pages x 24 granules (every block eligible): bound drops to 48
    a.observe(t, np.array([[48, chunk]], np.uint32))
    assert a.stats()["used_bytes_bound"] == 48 * 256
    t2, up = a.reserve([0], [1])  # 48 + 32 <= 90 fits; without the observation 64 + 32 would not
    assert up == []
    # an observation taken before the latest reservation is ignored
    a.observe(t, np.array([[48, chunk]], np.uint32))
    assert a.stats()["used_bytes_bound"] == 80 * 256
    t3, up = a.reserve([0], [1])  # 80 + 32 > 90: next chunk
    assert up == [(0, chunk, 2 * chunk)]


def test_allocator_exact_reservation_and_room(kvz, oracle):
    """Exact reservations (the sizes the encoder will place) fill a chunk to the granule:
    the oracle encodes pages into the cursor the allocator hands out, page runs split at
    the chunk's room, and the device cursor equals the allocator's bound after each run."""
    cfg = kvgen.KVConfig("alloc-exact", 1, 2, 8, 2, 20, seed=23, block_outlier_frac=0.3)
    hkv = cfg.hkv
    pool = kvgen.bits(kvgen.gen_pages(cfg, 20))
    chunk = 256  # 4..5 pages of 52..64 granules
    a = kvz.Allocator(arena_bytes=chunk * 256 * 16, chunk_granules=chunk, num_cursors=1, num_kv_heads=hkv)
    assert a.room(0) == 0
    # exact sizes of each page from the oracle's own encode (12 or 16 granules per group)
    sizes = []
    for p in range(20):
        g = 0
        for h in range(hkv):
            for kv in range(2):
                for j in range(4):
                    g += 3 if oracle.encode_block(pool[p, h, kv], bool(kv), j)[1] != 0xFF else 4
        sizes.append(g)
    meta = np.zeros((20, hkv, 2), np.uint64)
    arena = np.zeros(chunk * 256 * 16, np.uint8)
    cur = np.zeros((1, 2), np.uint32)
    p, runs = 0, 0
    while p < 20:
        room = a.room(0)
        q, tot = p, 0
        while q < 20 and tot + sizes[q] <= room:
            tot += sizes[q]
            q += 1
        if q == p:  # nothing fits the current chunk: the run opens a fresh one
            while q < 20 and tot + sizes[q] <= chunk:
                tot += sizes[q]
                q += 1
        t, up = a.reserve_granules([0], [tot])
        for c, pos, end in up:
            cur[c] = (pos, end)
        src = np.arange(p, q, dtype=np.int32)
        assert oracle.encode_pages(pool, src, src, np.zeros(q - p, np.int32), meta, arena, cur, hkv) == 0
        assert int(cur[0, 1]) - int(cur[0, 0]) == a.room(0)  # allocator bound == device cursor
        p, runs = q, runs + 1
    # every chunk but the last is left only when the next page no longer fits it
    held = a.stats()["chunks_held"]
    assert held * chunk - sum(sizes) < held * max(sizes) + chunk
    out, st = oracle.decode_pages(meta, arena, np.arange(20, dtype=np.int32), hkv)
    assert st == 0 and np.array_equal(out, pool)
    with pytest.raises(kvz.KvzError):
        a.reserve_granules([0], [chunk + 1])  # more than a chunk


def test_allocator_with_oracle_stream(kvz, oracle):
    """Streaming page completions for several sequences, the oracle encoding into the
    cursors the allocator hands out: no group ever overflows, chunks are recycled."""
    cfg = kvgen.KVConfig("alloc-sim", 1, 4, 8, 2, 24, seed=21, block_outlier_frac=0.3)
    hkv = cfg.hkv
    pool = kvgen.bits(kvgen.gen_pages(cfg, 24))
    chunk = 5 * 64  # 5 worst-case pages per chunk
    nchunks = 12
    arena = np.zeros(nchunks * chunk * 256, np.uint8)
    a = kvz.Allocator(arena.size, chunk, num_cursors=cfg.batch, num_kv_heads=hkv)
    cursors = np.zeros((cfg.batch, 2), np.uint32)
    meta = np.zeros((200, hkv, 2), np.uint64)
    next_meta = 0
    owner = {}
    for step in range(12):
        seqs = [s for s in range(cfg.batch) if (step + s) % 3 != 0]
        pages = [1 + (s % 2) for s in seqs]
        t, ups = a.reserve(seqs, pages)
        for c, pos, end in ups:
            cursors[c] = (pos, end)
        src, dst, dseq = [], [], []
        for s, n in zip(seqs, pages):
            for _ in range(n):
                src.append((step * 7 + s * 5 + len(src)) % 24)
                dst.append(next_meta)
                owner[next_meta] = s
                next_meta += 1
                dseq.append(s)
        st = oracle.encode_pages(pool, src, dst, dseq, meta, arena, cursors, hkv)
        assert st == 0, step
        a.observe(t, cursors)
        if step == 6:  # sequence 1 finishes; its chunks go back to the pool
            a.release(1)
            cursors[1] = (0, 0)
            for m_id in [k for k, v in owner.items() if v == 1]:
                meta[m_id] = 0
                owner.pop(m_id)
    # every recorded group lies inside a chunk and no two groups overlap
    spans = []
    for m_id in owner:
        for h in range(hkv):
            for kv in range(2):
                w = int(meta[m_id, h, kv])
                off = w & 0xFFFFFFFF
                size = sum(4 if (w >> (32 + 8 * j)) & 0xFF == 0xFF else 3 for j in range(4))
                assert off // chunk == (off + size - 1) // chunk
                spans.append((off, off + size))
    spans.sort()
    assert all(spans[k][1] <= spans[k + 1][0] for k in range(len(spans) - 1))
    st = a.stats()
    assert st["chunks_held"] + st["chunks_free"] == nchunks


def test_allocator_random_exact_reservations_model(kvz):
    """Random exact reservations and releases over a small arena, against a model of the
    device cursors: every granted region lies in one chunk owned by its cursor, regions of
    live cursors never overlap, the allocator's room equals the model cursor's room, a
    refused reservation changes nothing, and releasing every cursor frees every chunk."""
    rng = np.random.default_rng(7)
    chunk, nchunks, ncur = 64, 12, 6
    a = kvz.Allocator(arena_bytes=chunk * 256 * nchunks, chunk_granules=chunk, num_cursors=ncur, num_kv_heads=2)
    cur = {}  # cursor -> [pos, end] in granules (the device cursor after the updates)
    regions = {c: [] for c in range(ncur)}
    refused = 0
    for _ in range(3000):
        if rng.random() < 0.12:
            c = int(rng.integers(ncur))
            a.release(c)
            regions[c] = []
            cur.pop(c, None)
            assert a.room(c) == 0
        else:
            ids = rng.choice(ncur, size=int(rng.integers(1, 4)), replace=False).astype(np.int32)
            gr = rng.integers(1, chunk + 1, size=ids.size).astype(np.uint64)
            before = a.stats()
            try:
                _, ups = a.reserve_granules(ids, gr)
            except kvz.KvzError as e:
                assert e.code == kvz.ERR_OUT_OF_SPACE
                assert a.stats() == before
                refused += 1
                continue
            for c, pos, end in ups:
                cur[c] = [pos, end]
            for c, g in zip(ids.tolist(), gr.tolist()):
                pos, end = cur[c]
                assert pos + g <= end and end - pos <= chunk
                assert pos // chunk == (pos + g - 1) // chunk  # inside one chunk
                regions[c].append((pos, pos + g))
                cur[c][0] = pos + g
        st = a.stats()
        assert st["chunks_held"] + st["chunks_free"] == nchunks
        assert st["held_bytes"] == st["chunks_held"] * chunk * 256
        for c in range(ncur):
            assert a.room(c) == (cur[c][1] - cur[c][0] if c in cur else 0)
        live = sorted((r, c) for c in range(ncur) for r in regions[c])
        for (r0, c0), (r1, c1) in zip(live, live[1:]):
            assert r0[1] <= r1[0], (r0, c0, r1, c1)
        chunks_of = {c: {r[0] // chunk for r in regions[c]} for c in range(ncur)}
        for c0 in range(ncur):
            for c1 in range(c0 + 1, ncur):
                assert not (chunks_of[c0] & chunks_of[c1])  # a chunk belongs to one cursor
    assert refused > 0  # the arena did run out along the way
    for c in range(ncur):
        a.release(c)
    assert a.stats()["chunks_free"] == nchunks
