"""Pins of the group-adaptive additive tile oracle (oracle/oga.c) against what the GAAC
page fixes: Table 9's byte budget, the mode rule and escape sizes of "Group-adaptive
additive coding", the window calibration of "Contiguous exponent concentration",
hand-worked tiles (tests/golden/ga_examples.txt), losslessness, and the storage classes
of "Block-Wise Compression Scheduling"."""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x) -> np.ndarray:
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _golden():
    cases = []
    with open(os.path.join(GOLDEN, "ga_examples.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            name, *fields = line.split()
            spec = dict(f.split("=", 1) for f in fields)
            cases.append(pytest.param(spec, id=name))
    return cases


def _tile_from_spec(spec):
    page = np.full((16, 128), int(spec["fill"], 16), np.uint16)
    for item in spec["set"].split(","):
        t, d, v = item.split(":")
        page[int(t), int(d)] = int(v, 16)
    b3 = np.full(128, int(spec["b3"]), np.uint8)
    b4 = np.full(128, int(spec["b4"]), np.uint8)
    return page, spec["kind"] == "V", b3, b4


def _expand(field, count, width, base):
    """'k:v,...,else:v' over `count` items of `width` bytes (dot-separated hex) -> bytes."""
    out = np.zeros(count * width, np.uint8)
    default, sets = None, {}
    for item in field.split(","):
        k, v = item.split(":")
        vals = [int(x, 16) for x in v.split(".")]
        if k == "else":
            default = vals
        else:
            sets[int(k)] = vals
    for n in range(count):
        vals = sets.get(n, default)
        out[n * width:(n + 1) * width] = vals
    return out


@pytest.mark.parametrize("spec", _golden())
def test_golden_tiles(oracle, spec):
    page, is_v, b3, b4 = _tile_from_spec(spec)
    data = np.frombuffer(oracle.ga_encode_tile(page, is_v, b3, b4), np.uint8)
    assert data.size == int(spec["size"])
    if data.size == oracle.GA_RAW:
        words = data.view("<u2")
        for item in spec["word"].split(","):
            k, v = item.split(":")
            assert words[int(k)] == int(v, 16)
    else:
        assert np.array_equal(data[:2048], _expand(spec["sf"], 2048, 1, 0))
        assert np.array_equal(data[2048:2816], _expand(spec["codes"], 256, 3, 0))
        assert np.array_equal(data[2816:2880], _expand(spec["tags"], 64, 1, 0))
        esc = bytes(int(x, 16) for x in spec["esc"].split(".")) if spec["esc"] else b""
        assert data[2880:2880 + len(esc)].tobytes() == esc
        assert not data[2880 + len(esc):].any()  # the rest of the escape slot is zero
    assert np.array_equal(oracle.ga_decode_tile(data.tobytes(), is_v, b3, b4), page)


def test_table9_byte_budget(oracle):
    """A tile whose groups all take the 3-bit mode: 2048 sign/fraction + 768 code + 64
    tag bytes = 11.25 bits per element, plus the 128-byte escape slot (32 mean + 96
    unused) = 3008 bytes; without fallback the raw tile is 4096 bytes."""
    page = np.full((16, 128), 0x3F80, np.uint16)
    data = oracle.ga_encode_tile(page, False, np.full(128, 127, np.uint8), np.full(128, 120, np.uint8))
    assert len(data) == 3008 == 2048 + 768 + 64 + 32 + 96
    assert (2048 + 768 + 64) * 8 / 2048 == 11.25
    assert 64 * 8 / 2048 == 2 / 8  # mode tags: 2 bits per 8-element group


@pytest.mark.parametrize(
    "e,b3,b4,mode",
    [
        ([120] * 8, 120, 100, 0),             # d3 = 0 everywhere
        ([127] * 8, 120, 100, 0),             # d3 = 7: top of the 8-wide window
        ([128] + [120] * 7, 120, 115, 1),     # d3 = 8 leaves the 3-bit window; d4 = 13
        ([130] + [115] * 7, 120, 115, 1),     # d3 < 0 for seven, all inside [115, 130]
        ([131] + [120] * 7, 120, 115, 2),     # d4 = 16: outside both
        ([119] + [120] * 7, 120, 120, 2),     # below both bases
        ([0] * 8, 0, 0, 0),
        ([255] * 8, 248, 240, 0),
        ([247] + [248] * 7, 248, 240, 1),
    ],
)
def test_mode_rule(oracle, e, b3, b4, mode):
    assert oracle.ga_group_mode(e, [b3] * 8, [b4] * 8) == mode


def test_mode_uses_each_elements_own_channel_bases(oracle):
    # element 3 has its own bases; the others would fit the 3-bit window
    b3, b4 = [50] * 8, [40] * 8
    b3[3], b4[3] = 200, 190
    e = [52] * 8
    e[3] = 205
    assert oracle.ga_group_mode(e, b3, b4) == 0
    e[3] = 209  # 9 above its b3, 19 above its b4
    assert oracle.ga_group_mode(e, b3, b4) == 2


def _positions(oracle, is_v):
    """(token, dim) of element i of group q, from the storage order of the 12-bit format."""
    pos = {}
    for L in range(32):
        for j in range(4):
            for f in range(2):
                q = 8 * L + 2 * j + f
                pos[q] = [oracle.block_position(is_v, j, L, f, i) for i in range(8)]
    return pos


@pytest.mark.parametrize("is_v", [False, True])
@pytest.mark.parametrize("mode,n", [(1, 128), (1, 129), (2, 25), (2, 26)])
def test_escape_slot_capacity(oracle, is_v, mode, n):
    """A 4-bit group adds one escape byte, a raw group five; a tile fits its 3008-byte
    slot while the escape bytes fit in 128, else it is stored raw."""
    pos = _positions(oracle, is_v)
    page = np.full((16, 128), 0x3F80, np.uint16)  # e = 127
    b3, b4 = np.full(128, 124, np.uint8), np.full(128, 120, np.uint8)
    e_wide = 135 if mode == 1 else 20
    for q in range(0, 256, 256 // n if n <= 128 else 1)[:n]:
        t, d = pos[q][5]
        page[t, d] = e_wide << 7
    data = oracle.ga_encode_tile(page, is_v, b3, b4)
    escape = n * (1 if mode == 1 else 5)
    assert len(data) == (3008 if escape <= 128 else 4096)
    if len(data) == 3008:
        tags = np.frombuffer(data[2816:2880], np.uint8)
        modes = [(tags[q // 4] >> (2 * (q % 4))) & 3 for q in range(256)]
        assert sum(m == mode for m in modes) == n and sum(m != 0 for m in modes) == n
    assert np.array_equal(oracle.ga_decode_tile(data, is_v, b3, b4), page)


def _channel_pages(values_per_channel):
    """[n][16][128] pages whose channel c holds values_per_channel[c] (exponents) over tokens."""
    n_tok = max(len(v) for v in values_per_channel.values())
    n = (n_tok + 15) // 16
    pages = np.full((n * 16, 128), 0, np.uint16)
    fill = {}
    for c, exps in values_per_channel.items():
        col = list(exps) + [exps[-1]] * (n * 16 - len(exps))
        fill[c] = col
        pages[:, c] = np.array(col, np.uint16) << 7
    return pages.reshape(n, 16, 128), fill


def test_calibration_windows(oracle):
    chans = {
        0: [127] * 16,                         # one exponent: lowest windows holding it
        1: [100] * 10 + [108] * 9 + [100] * 13,  # 8-window ties between starts 93..100 -> 93
        2: [255] * 16,                         # windows end at 255
        3: [0] * 16,
        4: [60] * 3 + [70] * 20 + [71] * 9,    # 8-window: 70..71 = 29 beats 60 (3); 16: 60..71
    }
    pages, fill = _channel_pages(chans)
    b3, b4 = oracle.ga_calibrate(pages)
    assert (b3[0], b4[0]) == (120, 112)
    assert (b3[1], b4[1]) == (93, 93)
    assert (b3[2], b4[2]) == (248, 240)
    assert (b3[3], b4[3]) == (0, 0)
    assert (b3[4], b4[4]) == (64, 56)
    # channels 5..127 hold exponent 0 only (the page default)
    assert not b3[5:].any() and not b4[5:].any()


def test_calibration_coverage_brute_force(oracle):
    """On small random samples, the chosen windows cover the most values of all
    windows of their width (checked by counting each window)."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((2, 16, 128)) * np.exp2(rng.integers(-6, 6, 128))).astype(np.float32)
    pages = _bf16(x)
    b3, b4 = oracle.ga_calibrate(pages)
    e = ((pages >> 7) & 0xFF).reshape(-1, 128).astype(np.int64)
    for c in range(0, 128, 7):
        for w, b in ((8, b3[c]), (16, b4[c])):
            cover = [np.sum((e[:, c] >= s) & (e[:, c] < s + w)) for s in range(0, 257 - w)]
            assert cover[b] == max(cover) and cover.index(max(cover)) == b


@pytest.mark.parametrize("is_v", [False, True])
def test_lossless_on_adversarial_values(oracle, is_v):
    """Every BF16 pattern comes back (zeros, subnormals, inf, NaN, both signs), whatever
    the bases: a mismatch only costs size."""
    rng = np.random.default_rng(11)
    for trial in range(6):
        page = rng.integers(0, 1 << 16, (16, 128), dtype=np.uint16)
        if trial % 2:
            page[:, ::3] = rng.choice(np.array([0x0000, 0x8000, 0x0001, 0x7F80, 0xFF80, 0x7FC0, 0x807F], np.uint16),
                                      (16, 43))
        b3 = rng.integers(0, 249, 128).astype(np.uint8)
        b4 = rng.integers(0, 241, 128).astype(np.uint8)
        data = oracle.ga_encode_tile(page, is_v, b3, b4)
        assert np.array_equal(oracle.ga_decode_tile(data, is_v, b3, b4), page)


@pytest.mark.parametrize("is_v", [False, True])
def test_sign_fraction_bytes_follow_storage_order(oracle, is_v):
    rng = np.random.default_rng(5)
    page = _bf16(rng.standard_normal((16, 128)) * 0.1)
    b3, b4 = oracle.ga_calibrate(page[None])
    data = np.frombuffer(oracle.ga_encode_tile(page, is_v, b3, b4), np.uint8)
    assert data.size == 3008
    for L, j, f, i in [(0, 0, 0, 0), (5, 1, 1, 3), (31, 3, 1, 7), (17, 2, 0, 6)]:
        t, d = oracle.block_position(is_v, j, L, f, i)
        w = int(page[t, d])
        assert data[512 * j + 16 * L + 8 * f + i] == ((w >> 8) & 0x80) | (w & 0x7F)


def test_pages_two_storage_classes_and_cursors(oracle):
    """Entries: 31-bit granule offset + raw bit; tiles are appended at the sequence
    cursor in (page, head, K|V) order; 47 granules compressed, 64 raw."""
    hkv = 2
    rng = np.random.default_rng(8)
    pool = _bf16(rng.standard_normal((3, hkv, 2, 16, 128)) * 0.05)
    pool[1, 1, 0, :, 0::2] = 0x3580 | np.uint16(0)  # far below the windows: many raw groups
    pool[1, 1, 0, :, 1::2] = 0x7F00
    bases = oracle.ga_calibrate_pool(pool, [0, 2], hkv)
    meta = np.zeros((4, hkv, 2), np.uint32)
    arena = np.zeros(64 * 1000, np.uint8)
    cur = np.array([[10, 1000]], np.uint32)
    st = oracle.ga_encode_pages(pool, bases, [0, 1], [3, 0], [0, 0], meta, arena, cur, hkv)
    assert st == 0
    sizes = []
    for p in (3, 0):
        for h in range(hkv):
            for kv in range(2):
                sizes.append(64 if meta[p, h, kv] & oracle.GA_ENTRY_RAW else 47)
    offs = [int(meta[p, h, kv]) & 0x7FFFFFFF for p in (3, 0) for h in range(hkv) for kv in range(2)]
    assert offs == list(10 + np.concatenate([[0], np.cumsum(sizes)[:-1]]))
    assert meta[0, 1, 0] & oracle.GA_ENTRY_RAW  # the planted tile fell back to raw
    assert int(cur[0, 0]) == 10 + sum(sizes)
    out, st = oracle.ga_decode_pages(meta, arena, bases, [3, 0], hkv)
    assert st == 0 and np.array_equal(out, pool[[0, 1]])


def test_pages_arena_full_and_bad_index(oracle):
    hkv = 1
    pool = np.full((2, hkv, 2, 16, 128), 0x3F80, np.uint16)
    bases = oracle.ga_calibrate_pool(pool, [0], hkv)
    meta = np.zeros((2, hkv, 2), np.uint32)
    arena = np.zeros(64 * 100, np.uint8)
    cur = np.array([[0, 100]], np.uint32)  # room for two 47-granule tiles, not three
    st = oracle.ga_encode_pages(pool, bases, [0, 1], [0, 1], [0, 0], meta, arena, cur, hkv)
    assert st == 1  # arena full
    assert meta[0, 0, 0] == 0 and meta[0, 0, 1] == 47
    assert meta[1, 0, 0] == oracle.GA_ENTRY_INVALID and meta[1, 0, 1] == oracle.GA_ENTRY_INVALID
    _, st = oracle.ga_decode_pages(meta, arena, bases, [1], hkv)
    assert st == 8  # bad metadata
    before = meta.copy()
    st = oracle.ga_encode_pages(pool, bases, [0, 5], [0, 1], [0, 0], meta, arena, cur, hkv)
    assert st == 2 and np.array_equal(meta, before)  # a bad index makes the call a no-op


def test_ga_attention_equals_raw_attention(oracle):
    """Tiles are lossless, so attention over tiles + raw tail equals attention over the
    plain pages, bit for bit in the fp64 oracle (the same arithmetic after decode)."""
    hkv, hq, B = 2, 8, 3
    rng = np.random.default_rng(21)
    n_pool = 12
    pool = _bf16(rng.standard_normal((n_pool, hkv, 2, 16, 128)) * 0.3)
    pool[4, 0, 1, :, 5] = 0x3580  # a few raw groups
    q = _bf16(rng.standard_normal((B, hq, 128)))
    seq_lens = np.array([16 * 3 + 5, 16 * 2, 7], np.int32)
    table = np.array([[0, 1, 2, 9], [3, 4, -1, -1], [10, -1, -1, -1]], np.int32)
    bases = oracle.ga_calibrate_pool(pool, [0, 1, 2, 3], hkv)
    meta = np.zeros((n_pool, hkv, 2), np.uint32)
    arena = np.zeros(64 * 64 * 40, np.uint8)
    cur = np.array([[0, 64 * 40]], np.uint32)
    full = [0, 1, 2, 3, 4]
    assert oracle.ga_encode_pages(pool, bases, full, full, [0] * 5, meta, arena, cur, hkv) == 0
    tail = np.array([9, -1, 10], np.int32)
    ref, st = oracle.attention_raw(q, table, seq_lens, pool, hkv)
    assert st == 0
    got, st = oracle.ga_decode_attention(q, table, seq_lens, tail, meta, arena, bases, pool, hkv)
    assert st == 0
    assert np.array_equal(got, ref)
