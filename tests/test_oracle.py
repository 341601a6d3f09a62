"""Pins for the CPU oracle: each test checks it against something other than itself.

What pins what (page titles, sections):
  * block sizes 768 / 1024 B and 8 B of group metadata   -- ZipFusion "How it works" step 3,
    metadata paragraph (closed form from the bit counts);
  * e = b + 2d + r restore, over all 65536 BF16 words    -- ZipFusion step 4 (round trips of
    every word, alone and beside a partner at every allowed distance);
  * eligibility window [b, b+15], b = even floor of min   -- ZipFusion step 2 (closed form by
    parity of the minimum, over every (min, max) pair);
  * zeros / subnormals / inf / NaN                       -- the literal step-2 rule;
  * byte-add restore (mask one branch, unpack the other,
    one 32-bit add of b/2 per byte, no carry)             -- ZipFusion layout paragraph, applied
    to the oracle's bytes and gathered with the tensor-core fragment table below;
  * K / V operand-role layouts                           -- ZipFusion layout paragraph: the
    stored lane fragments must be the m16n8k16 A operands of K (QK^T) and of V^T (PV);
  * BF16 fields and value formula                        -- ExANS "Under the hood";
  * attention                                             -- GAAC "Attention with On-the-Fly
    Decompression" (one softmax over compressed pages and raw tail): torch SDPA in
    float64, one-token and identical-key closed forms.
"""
import math
import os

import numpy as np
import pytest
import torch

import kvgen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------------------
# tensor-core A-operand fragment table for mma.m16n8k16 (PTX ISA, "Matrix Fragments for
# mma.m16n8k16" with 16-bit A): register element a_i of a lane with groupID g and
# threadID_in_group t sits at row (g + ROW_OFF[i]) and column (2t + COL_OFF[i]).
# --------------------------------------------------------------------------------------
ROW_OFF = [0, 0, 8, 8, 0, 0, 8, 8]
COL_OFF = [0, 1, 0, 1, 8, 9, 8, 9]


def fragment_matrix(stored_lane_major: np.ndarray, f: int) -> np.ndarray:
    """16x16 A operand from storage-ordered values [32 lanes][2 frags][8]."""
    A = np.full((16, 16), -1, np.int64)
    for L in range(32):
        g, t = L // 4, L % 4
        for i in range(8):
            A[g + ROW_OFF[i], 2 * t + COL_OFF[i]] = stored_lane_major[L, f, i]
    return A


def storage_gather(page: np.ndarray, is_v: bool, j: int) -> np.ndarray:
    """Values of block j in storage order [32][2][8], gathered via the fragment table."""
    out = np.zeros((32, 2, 8), np.uint16)
    for L in range(32):
        g, t = L // 4, L % 4
        for f in range(2):
            for i in range(8):
                row, col = g + ROW_OFF[i], 2 * t + COL_OFF[i]
                if not is_v:  # K: A rows are tokens, columns dims of the 16-dim k-slice
                    out[L, f, i] = page[row, 32 * j + 16 * f + col]
                else:  # V^T: A rows are dims, columns tokens
                    out[L, f, i] = page[col, 32 * j + 16 * f + row]
    return out


def byte_add_restore(data: bytes, tag: int) -> np.ndarray:
    """Restore an eligible block with the byte trick: one masked branch, one unpacked
    branch, each plus b/2 replicated per byte.  Returns storage-ordered words [32][2][8]."""
    buf = np.frombuffer(data, np.uint8)
    low = buf[:512].reshape(32, 2, 8).astype(np.uint32)
    W = buf[512:768].copy().view("<u4").reshape(32, 2).astype(np.uint64)
    bb = np.uint64(tag * 0x01010101)
    h_lo = ((W & 0x87878787) + bb) & 0xFFFFFFFF
    h_hi = ((((W >> 4) & 0x07070707) | ((W << 4) & 0x80808080)) + bb) & 0xFFFFFFFF
    high = np.zeros((32, 2, 8), np.uint32)
    for k in range(4):
        high[:, :, k] = (h_lo >> np.uint64(8 * k)) & 0xFF
        high[:, :, k + 4] = (h_hi >> np.uint64(8 * k)) & 0xFF
    return ((high << 8) | low).astype(np.uint16)


def page_with(fill: int, sets=()) -> np.ndarray:
    p = np.full((16, 128), fill, np.uint16)
    for tok, dim, w in sets:
        p[tok, dim] = w
    return p


def fields(w):
    return (w >> 15) & 1, (w >> 7) & 0xFF, w & 0x7F


# --------------------------------------------------------------------------------------
# sizes and golden examples
# --------------------------------------------------------------------------------------
def test_block_sizes_closed_form(oracle):
    # 512 values x (8 kept + 4 code) bits = 768 B; raw = 512 x 16 bits = 1024 B
    elig = page_with(0x3F80)
    data, tag = oracle.encode_block(elig, False, 0)
    assert len(data) == 512 * (8 + 4) // 8 == 768 and tag == 127 // 2
    raw = page_with(0x3F80, [(0, 0, 0x4580), (1, 1, 0x3780)])
    data, tag = oracle.encode_block(raw, False, 0)
    assert len(data) == 512 * 16 // 8 == 1024 and tag == 0xFF


def _parse_examples():
    rows = []
    with open(os.path.join(GOLDEN, "block_examples.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, *kvs = line.split()
            d = dict(kv.split("=", 1) for kv in kvs)
            rows.append((name, d))
    return rows


def _idxmap(spec: str, n: int) -> np.ndarray:
    out = np.zeros(n, np.int64)
    for part in spec.split(","):
        k, v = part.split(":")
        if k == "else":
            out[:] = int(v, 0)
    for part in spec.split(","):
        k, v = part.split(":")
        if k != "else":
            out[int(k)] = int(v, 0)
    return out


@pytest.mark.parametrize("name,spec", _parse_examples())
def test_golden_block_examples(oracle, name, spec):
    sets = []
    for s in spec["set"].split(","):
        tok, dim, w = s.split(":")
        sets.append((int(tok), int(dim), int(w, 0)))
    page = page_with(int(spec["fill"], 0), sets)
    is_v = spec["kind"] == "V"
    j = int(spec["block"])
    data, tag = oracle.encode_block(page, is_v, j)
    assert tag == int(spec["tag"]) and len(data) == int(spec["size"])
    buf = np.frombuffer(data, np.uint8)
    if "low" in spec:
        assert np.array_equal(buf[:512], _idxmap(spec["low"], 512).astype(np.uint8))
        assert np.array_equal(buf[512:], _idxmap(spec["code"], 256).astype(np.uint8))
    else:
        words = buf.view("<u2")
        assert np.array_equal(words, _idxmap(spec["word"], 512).astype(np.uint16))
    back = oracle.decode_block(data, tag, is_v, j, np.zeros((16, 128), np.uint16))
    assert np.array_equal(back[:, 32 * j: 32 * j + 32], page[:, 32 * j: 32 * j + 32])


def test_golden_bf16_fields(oracle):
    with open(os.path.join(GOLDEN, "bf16_fields.txt")) as fh:
        rows = [ln.split() for ln in fh if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 6
    for word, s, e, f, val, E, SF in rows:
        w = int(word, 16)
        assert fields(w) == (int(s), int(e), int(f))
        assert oracle.bf16_exponent(w) == int(e)
        assert oracle.bf16_value(w) == float(val)
        # ExANS byte streams and their reassembly
        assert (w >> 7) & 0xFF == int(E, 16)
        assert (((w >> 8) & 0x80) | (w & 0x7F)) == int(SF, 16)


# --------------------------------------------------------------------------------------
# field formulas over every word
# --------------------------------------------------------------------------------------
def test_exans_field_split_and_value_formula_all_words(oracle):
    w = np.arange(65536, dtype=np.int64)
    E = (w >> 7) & 0xFF
    SF = ((w >> 8) & 0x80) | (w & 0x7F)
    word = ((SF & 0x80) << 8) | (E << 7) | (SF & 0x7F)
    assert np.array_equal(word, w)
    vals = torch.from_numpy(w.astype(np.int16)).view(torch.bfloat16).double().numpy()
    s, e, f = (w >> 15) & 1, (w >> 7) & 0xFF, w & 0x7F
    normal = (e > 0) & (e < 255)
    formula = np.where(s == 1, -1.0, 1.0) * np.exp2(e - 127.0) * (1 + f / 128.0)
    assert np.array_equal(vals[normal], formula[normal])
    for x in (0x0000, 0x8000, 0x0001, 0x3F80, 0x7F80, 0xFF80, 0x7FC1, 0x8123):
        got = oracle.bf16_value(x)
        ref = float(torch.tensor([x if x < 32768 else x - 65536], dtype=torch.int16).view(torch.bfloat16))
        assert (math.isnan(got) and math.isnan(ref)) or got == ref


# --------------------------------------------------------------------------------------
# exhaustive round trips and the eligibility boundary
# --------------------------------------------------------------------------------------
def test_every_word_alone_round_trips(oracle):
    """A block holding one repeated word has spread 0: always eligible, tag = e // 2."""
    for w in range(65536):
        page = np.full((16, 128), w, np.uint16)
        j = w % 4
        is_v = bool(w & 4)
        data, tag = oracle.encode_block(page, is_v, j)
        e = (w >> 7) & 0xFF
        assert tag == e // 2 and len(data) == 768, hex(w)
        back = oracle.decode_block(data, tag, is_v, j)
        assert np.all(back[:, 32 * j: 32 * j + 32] == w), hex(w)


def test_every_word_beside_partner_round_trips(oracle):
    """Word w together with a partner whose exponent is the block minimum, at every
    distance 0..17: eligibility follows the window rule and every bit comes back."""
    rng = np.random.default_rng(7)
    for w in range(0, 65536, 3):
        s, e, f = fields(w)
        for dist in (0, 1, 14, 15, 16, 17):
            m = e - dist
            if m < 0:
                continue
            partner = (int(rng.integers(0, 2)) << 15) | (m << 7) | int(rng.integers(0, 128))
            page = np.full((16, 128), partner, np.uint16)
            page[int(rng.integers(0, 16)), 32 + int(rng.integers(0, 32))] = w
            data, tag = oracle.encode_block(page, bool(w & 1), 1)
            eligible = (dist <= 15) if m % 2 == 0 else (dist <= 14)
            assert (tag != 0xFF) == eligible, (hex(w), dist)
            if eligible:
                assert tag == m // 2
            back = oracle.decode_block(data, tag, bool(w & 1), 1)
            assert np.array_equal(back[:, 32:64], page[:, 32:64])


def test_eligibility_boundary_every_min_max(oracle):
    """Every (min, max) exponent pair with max - min <= 17: eligible iff, for an even
    minimum, max - min <= 15 and, for an odd minimum, max - min <= 14."""
    for mn in range(256):
        for mx in range(mn, min(255, mn + 17) + 1):
            page = np.full((16, 128), (mn << 7) | 0x15, np.uint16)
            page[9, 100] = 0x8000 | (mx << 7) | 0x2A
            data, tag = oracle.encode_block(page, False, 3)
            expect = (mx - mn <= 15) if mn % 2 == 0 else (mx - mn <= 14)
            assert (tag != 0xFF) == expect, (mn, mx)
            assert len(data) == (768 if expect else 1024)


def test_special_values(oracle):
    zero, nzero = 0x0000, 0x8000
    # all-zero block: every exponent is 0 -> eligible with b = 0; signs survive
    page = np.zeros((16, 128), np.uint16)
    page[::2, ::3] = nzero
    data, tag = oracle.encode_block(page, True, 2)
    assert tag == 0 and len(data) == 768
    assert np.array_equal(oracle.decode_block(data, tag, True, 2)[:, 64:96], page[:, 64:96])
    # subnormals and zeros share exponent 0 -> eligible
    page = np.full((16, 128), 0x0001, np.uint16)
    page[3, 5] = 0x807F
    page[4, 6] = zero
    data, tag = oracle.encode_block(page, False, 0)
    assert tag == 0 and np.array_equal(oracle.decode_block(data, tag, False, 0)[:, :32], page[:, :32])
    # one zero among ordinary values (e ~ 127) breaks the window -> raw
    page = np.full((16, 128), 0x3F80, np.uint16)
    page[0, 0] = nzero
    data, tag = oracle.encode_block(page, False, 0)
    assert tag == 0xFF
    assert np.array_equal(oracle.decode_block(data, tag, False, 0)[:, :32], page[:, :32])
    # one NaN among ordinary values -> raw, payload kept
    page[0, 0] = 0x7FC5
    data, tag = oracle.encode_block(page, False, 0)
    assert tag == 0xFF and oracle.decode_block(data, tag, False, 0)[0, 0] == 0x7FC5
    # inf, NaN and huge values together: exponents 240..255 -> b = 240, eligible
    page = np.full((16, 128), 0x7800, np.uint16)  # e = 240
    page[1, 1], page[2, 2], page[3, 3] = 0x7F80, 0xFF80, 0xFFC3  # +inf, -inf, NaN
    data, tag = oracle.encode_block(page, False, 0)
    assert tag == 120
    assert np.array_equal(oracle.decode_block(data, tag, False, 0)[:, :32], page[:, :32])


def test_invalid_tags_rejected(oracle):
    data, tag = oracle.encode_block(page_with(0x3F80), False, 0)
    for bad in (0x80, 0x9A, 0xFE):
        with pytest.raises(ValueError):
            oracle.decode_block(data, bad, False, 0)


# --------------------------------------------------------------------------------------
# the byte-add restore and the operand-role layouts
# --------------------------------------------------------------------------------------
def test_byte_add_never_carries_exhaustive():
    """High byte = sign<<7 | (b/2 + d) from one add, for every sign, b/2 and d with
    b/2 + d <= 127 (e = b + 2d + r <= 255), on both branches and all four byte lanes."""
    s = np.arange(2)[:, None, None]
    h = np.arange(128)[None, :, None]
    d = np.arange(8)[None, None, :]
    ok = (h + d) <= 127
    lo_code = (s << 7) | d                      # k-side of a code byte
    hi_code = (s << 3) | (d << 4)               # (k+4)-side of a code byte
    assert np.all((((lo_code & 0x87) + h) == ((s << 7) | (h + d)))[np.broadcast_to(ok, (2, 128, 8))])
    swapped = ((hi_code >> 4) & 0x07) | ((hi_code << 4) & 0x80)
    assert np.all(((swapped + h) == ((s << 7) | (h + d)))[np.broadcast_to(ok, (2, 128, 8))])
    # four lanes at once: random per-lane (s, d) under one h, sum stays per byte
    rng = np.random.default_rng(1)
    for hv in range(128):
        n = 4096
        ss = rng.integers(0, 2, (n, 4))
        dd = rng.integers(0, min(7, 127 - hv) + 1, (n, 4))
        bytes_ = (ss << 7) | dd
        W = (bytes_ * (256 ** np.arange(4))).sum(1).astype(np.uint64)
        out = ((W & 0x87878787) + np.uint64(hv * 0x01010101)) & 0xFFFFFFFF
        want = (((ss << 7) | (dd + hv)) * (256 ** np.arange(4))).sum(1).astype(np.uint64)
        assert np.array_equal(out, want)


def test_byte_add_restore_matches_oracle_bytes(oracle):
    """The oracle's eligible blocks, restored with the byte trick and laid out with the
    fragment table, reproduce the input words."""
    cfg = kvgen.C0
    pool = kvgen.bits(kvgen.gen_pages(cfg, 6))
    seen = 0
    for p in range(6):
        for h in range(cfg.hkv):
            for kv in range(2):
                for j in range(4):
                    page = pool[p, h, kv]
                    data, tag = oracle.encode_block(page, bool(kv), j)
                    if tag == 0xFF:
                        continue
                    seen += 1
                    got = byte_add_restore(data, tag)
                    assert np.array_equal(got, storage_gather(page, bool(kv), j))
    assert seen > 20


def test_layouts_are_tensor_core_operands(oracle):
    """Raw blocks keep words in storage order, so a raw block exposes the layout itself:
    each lane's eight words of fragment f must form the 16x16 A operand of the block's
    role -- K[tokens][16 dims] for QK^T, V^T[16 dims][tokens] for PV."""
    rng = np.random.default_rng(3)
    for is_v in (False, True):
        for j in range(4):
            page = rng.integers(0, 65536, (16, 128)).astype(np.uint16)
            page[0, :] = 0x7F80  # inf + ordinary values -> raw
            page[1, :] = 0x0001
            data, tag = oracle.encode_block(page, is_v, j)
            assert tag == 0xFF
            stored = np.frombuffer(data, "<u2").reshape(32, 2, 8)
            for f in range(2):
                A = fragment_matrix(stored, f)
                dims = slice(32 * j + 16 * f, 32 * j + 16 * f + 16)
                want = page[:, dims].T if is_v else page[:, dims]
                assert np.array_equal(A, want.astype(np.int64)), (is_v, j, f)


def test_block_position_is_bijection(oracle):
    for is_v in (False, True):
        for j in range(4):
            seen = set()
            for L in range(32):
                for f in range(2):
                    for i in range(8):
                        tok, dim = oracle.block_position(is_v, j, L, f, i)
                        assert 0 <= tok < 16 and 32 * j <= dim < 32 * j + 32
                        seen.add((tok, dim))
            assert len(seen) == 512


# --------------------------------------------------------------------------------------
# page encode: placement, metadata bytes, cursors, errors
# --------------------------------------------------------------------------------------
def _encode_setup(oracle, cfg, n_pages, cursors_spec, arena_bytes=1 << 22):
    pool = kvgen.bits(kvgen.gen_pages(cfg, n_pages))
    meta = np.zeros((n_pages, cfg.hkv, 2), np.uint64)
    arena = np.zeros(arena_bytes, np.uint8)
    cursors = np.array(cursors_spec, np.uint32).reshape(-1, 2)
    return pool, meta, arena, cursors


def test_encode_pages_tiles_cursor_regions(oracle):
    cfg = kvgen.C0
    n = 10
    pool, meta, arena, cursors = _encode_setup(oracle, cfg, n, [[4, 2000], [3000, 8000], [9000, 16000]])
    src = np.arange(n, dtype=np.int32)[::-1].copy()
    dst = np.arange(n, dtype=np.int32)
    seq = np.array([0, 0, 0, 1, 1, 1, 1, 2, 2, 2], np.int32)
    start = cursors[:, 0].copy()
    st = oracle.encode_pages(pool, src, dst, seq, meta, arena, cursors, cfg.hkv)
    assert st == 0
    # metadata bytes: 4-byte little-endian offset, then the four tags
    mb = meta.view(np.uint8).reshape(n, cfg.hkv, 2, 8)
    pos = start.astype(np.int64).copy()
    for p in range(n):
        for h in range(cfg.hkv):
            for kv in range(2):
                off = int(mb[dst[p], h, kv, :4].view("<u4")[0])
                tags = mb[dst[p], h, kv, 4:]
                assert off == pos[seq[p]]  # groups follow each other at the cursor
                at = off * 256
                for j in range(4):
                    size = 1024 if tags[j] == 0xFF else 768
                    data = arena[at: at + size].tobytes()
                    want, wtag = oracle.encode_block(pool[src[p], h, kv], bool(kv), j)
                    assert wtag == tags[j] and data == want
                    at += size
                pos[seq[p]] = at // 256
    assert np.array_equal(cursors[:, 0].astype(np.int64), pos)
    # and the whole thing decodes back to the pages
    back, st = oracle.decode_pages(meta, arena, dst, cfg.hkv)
    assert st == 0 and np.array_equal(back, pool[src])


def test_encode_pages_errors(oracle):
    cfg = kvgen.C0
    n = 4
    # decreasing cursor order -> no-op
    pool, meta, arena, cursors = _encode_setup(oracle, cfg, n, [[0, 4000], [4000, 8000]])
    before = cursors.copy()
    st = oracle.encode_pages(pool, np.arange(n), np.arange(n), [1, 1, 0, 0], meta, arena, cursors, cfg.hkv)
    assert st == oracle.BAD_ORDER and np.array_equal(cursors, before) and not meta.any()
    # index out of range -> no-op
    st = oracle.encode_pages(pool, [0, 1, 2, 9], np.arange(n), [0] * 4, meta, arena, cursors, cfg.hkv)
    assert st == oracle.BAD_INDEX and not meta.any() and not arena.any()
    # cursor region too small: groups past the end are not written, offset marked invalid
    pool, meta, arena, cursors = _encode_setup(oracle, cfg, n, [[0, 40]])
    st = oracle.encode_pages(pool, np.arange(n), np.arange(n), [0] * 4, meta, arena, cursors, cfg.hkv)
    assert st == oracle.ARENA_FULL
    offs = (meta & np.uint64(0xFFFFFFFF)).astype(np.int64).reshape(-1)
    sizes = [sum(3 if ((int(m) >> (32 + 8 * j)) & 0xFF) != 0xFF else 4 for j in range(4)) for m in meta.reshape(-1)]
    running = 0
    for o, s in zip(offs, sizes):
        if running + s <= 40:
            assert o == running
        else:
            assert o == 0xFFFFFFFF
        running += s
    assert cursors[0, 0] == running
    assert not arena[40 * 256:].any()


def test_decode_pages_bad_metadata(oracle):
    cfg = kvgen.C0
    pool, meta, arena, cursors = _encode_setup(oracle, cfg, 3, [[0, 4000]], arena_bytes=1 << 20)
    assert oracle.encode_pages(pool, [0, 1, 2], [0, 1, 2], [0, 0, 0], meta, arena, cursors, cfg.hkv) == 0
    bad = meta.copy()
    bad[1, 0, 1] = (bad[1, 0, 1] & np.uint64(0x00FFFFFFFFFFFFFF)) | np.uint64(0x85 << 56)
    bad[2, 1, 0] = np.uint64(0xFFFFFFFF) | (bad[2, 1, 0] & np.uint64(0xFFFFFFFF00000000))
    out, st = oracle.decode_pages(bad, arena, [0, 1, 2], cfg.hkv)
    assert st == oracle.BAD_META
    assert not out[1, 0, 1].any() and not out[2, 1, 0].any()
    assert np.array_equal(out[0], pool[0]) and np.array_equal(out[1, 0, 0], pool[1, 0, 0])


# --------------------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------------------
def _bf(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).double()


def _sdpa_reference(q, pool, table, seq_lens, hkv):
    B, hq, D = q.shape
    G = hq // hkv
    out = np.zeros((B, hq, D))
    for b in range(B):
        L = int(seq_lens[b])
        npg = (L + 15) // 16
        pages = pool[table[b, :npg]]  # [npg][hkv][2][16][128]
        K = _bf(pages[:, :, 0].transpose(1, 0, 2, 3).reshape(hkv, npg * 16, D)[:, :L])
        V = _bf(pages[:, :, 1].transpose(1, 0, 2, 3).reshape(hkv, npg * 16, D)[:, :L])
        Kx = K.repeat_interleave(G, 0)[None]
        Vx = V.repeat_interleave(G, 0)[None]
        o = torch.nn.functional.scaled_dot_product_attention(_bf(q[b])[None, :, None, :], Kx, Vx)
        out[b] = o[0, :, 0].numpy()
    return out


def _compressed_case(oracle, cfg, tail):
    lay = kvgen.gen_layout(cfg)
    table = lay["table"].numpy()
    seq_lens = lay["seq_lens"].numpy()
    pool = kvgen.bits(kvgen.gen_pages(cfg, cfg.num_pages))
    q = kvgen.bits(kvgen.gen_q(cfg))
    meta = np.zeros((cfg.num_pages, cfg.hkv, 2), np.uint64)
    arena = np.zeros(cfg.num_pages * cfg.hkv * 2 * 4096, np.uint8)
    full = table[:, : cfg.full_pages]
    seq = np.repeat(np.arange(cfg.batch, dtype=np.int32), cfg.full_pages)
    per = arena.size // 256 // cfg.batch
    cursors = np.array([[b * per, (b + 1) * per] for b in range(cfg.batch)], np.uint32)
    st = oracle.encode_pages(pool, full.reshape(-1), full.reshape(-1), seq, meta, arena, cursors, cfg.hkv)
    assert st == 0
    tail_page = table[:, cfg.full_pages] if tail else np.full(cfg.batch, -1, np.int32)
    return q, table, seq_lens, pool, meta, arena, tail_page


@pytest.mark.parametrize("cfg", [kvgen.C0, kvgen.C0_TAIL,
                                 kvgen.KVConfig("small-b3", 1, 3, 8, 2, 5, 1, 15, seed=11)])
def test_attention_matches_float64_sdpa(oracle, cfg):
    tail = cfg.tail_max > 0
    q, table, seq_lens, pool, meta, arena, tail_page = _compressed_case(oracle, cfg, tail)
    ref = _sdpa_reference(q, pool, table, seq_lens, cfg.hkv)
    out_c, st_c = oracle.decode_attention(q, table[:, : cfg.full_pages], seq_lens, tail_page, meta, arena, pool, cfg.hkv, nthreads=2)
    out_r, st_r = oracle.attention_raw(q, table, seq_lens, pool, cfg.hkv, nthreads=3)
    assert st_c == 0 and st_r == 0
    assert np.allclose(out_c, ref, rtol=1e-12, atol=1e-12)
    # compressed and raw oracle paths see the same BF16 values: identical results
    assert np.array_equal(out_c, out_r)


def test_attention_closed_forms(oracle):
    hkv, hq = 2, 8
    rng = np.random.default_rng(5)
    pool = rng.integers(0x3000, 0x4000, (4, hkv, 2, 16, 128)).astype(np.uint16)
    q = rng.integers(0x3000, 0x4000, (1, hq, 128)).astype(np.uint16)
    # one token: the output is that token's value row
    out, st = oracle.attention_raw(q, np.array([[2]]), np.array([1]), pool, hkv)
    assert st == 0
    for h in range(hq):
        assert np.array_equal(out[0, h], _bf(pool[2, h // 4, 1, 0]).numpy())
    # identical keys: uniform weights -> the mean of V
    same = pool.copy()
    same[:, :, 0] = pool[0, :, 0, :1]
    out, st = oracle.attention_raw(q, np.array([[0, 1, 3]]), np.array([40]), same, hkv)
    for h in range(hq):
        V = np.concatenate([_bf(same[p, h // 4, 1]).numpy() for p in (0, 1, 3)])[:40]
        assert np.allclose(out[0, h], V.mean(0), rtol=1e-13, atol=1e-15)
    # q = 0: also the mean of V
    out, st = oracle.attention_raw(np.zeros_like(q), np.array([[0, 1, 3]]), np.array([37]), pool, hkv)
    V = np.concatenate([_bf(pool[p, 1, 1]).numpy() for p in (0, 1, 3)])[:37]
    assert np.allclose(out[0, 7], V.mean(0), rtol=1e-13, atol=1e-15)
    # empty context: zero output
    out, st = oracle.attention_raw(q, np.array([[0]]), np.array([0]), pool, hkv)
    assert st == 0 and not out.any()


def test_attention_bad_meta_page_is_skipped(oracle):
    cfg = kvgen.C0
    q, table, seq_lens, pool, meta, arena, tail_page = _compressed_case(oracle, cfg, False)
    bad = meta.copy()
    victim = table[0, 5]
    bad[victim, 1, 0] = np.uint64(0xFFFFFFFF) | (bad[victim, 1, 0] & np.uint64(0xFFFFFFFF00000000))
    out, st = oracle.decode_attention(q, table, seq_lens, tail_page, bad, arena, pool, cfg.hkv)
    assert st == oracle.BAD_META
    keep = np.array([[p for p in table[0] if p != victim]], np.int32)
    ref1, _ = oracle.attention_raw(q, keep, np.array([seq_lens[0] - 16]), pool, cfg.hkv)
    ref0, _ = oracle.attention_raw(q, table, seq_lens, pool, cfg.hkv)
    G = cfg.hq // cfg.hkv
    assert np.array_equal(out[0, G:], ref1[0, G:])      # head group of KV head 1 loses the page
    assert np.array_equal(out[0, :G], ref0[0, :G])      # KV head 0 is untouched
    # missing tail page
    out, st = oracle.decode_attention(q, table, seq_lens + 3, np.full(1, -1, np.int32), meta, arena, pool, cfg.hkv)
    assert st & oracle.BAD_TAIL
