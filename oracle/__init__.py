"""CPU oracle for the 12-bit lossless BF16 KV format, the group-adaptive additive
tile format, and paged decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It wraps ``oref.c``, a
plain scalar C restatement of the ZipFusion 12-bit block format ("How it works",
steps 1-4, the operand-role layout and the metadata paragraphs) and of GQA decode
attention in double precision (GAAC, "Attention with On-the-Fly Decompression"),
and ``oga.c``, the GAAC group-adaptive additive codec ("Lossless KV Compression",
Table 9).  It shares no code with the CUDA library and never calls it.

Arrays are numpy arrays; BF16 values travel as ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboref.so")

ARENA_FULL = 1
BAD_INDEX = 2
BAD_ORDER = 4
BAD_META = 8
BAD_TAIL = 32

PAGE = 16
HEAD_DIM = 128


def build(force: bool = False) -> str:
    """Compile oref.c into liboref.so next to it (plain gcc, no CUDA)."""
    srcs = [os.path.join(_HERE, f) for f in ("oref.c", "oga.c", "of8.c")]
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= max(
        os.path.getmtime(f) for f in srcs + [os.path.join(_HERE, "oref.h")]
    ):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.check_call(
        ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-o", tmp, *srcs, "-lpthread", "-lm"]
    )
    os.replace(tmp, _SO)
    return _SO


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        P = ctypes.c_void_p
        i32, i64, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
        lib.oref_encode_block.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P]
        lib.oref_decode_block.argtypes = [P, ctypes.c_uint8, ctypes.c_int, ctypes.c_int, P]
        lib.oref_encode_pages.argtypes = [ctypes.c_int, P, i64, P, P, P, i32, P, i64, P, u64, P, i32]
        lib.oref_decode_pages.argtypes = [ctypes.c_int, P, i64, P, u64, P, i32, P]
        lib.oref_decode_attention.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int, P, P, P, i64, P, u64, P,
            i64, P, ctypes.c_int,
        ]
        lib.oref_attention_raw.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int, P, P, i64, P, ctypes.c_int,
        ]
        lib.oref_block_position.argtypes = [ctypes.c_int] * 5 + [P, P]
        lib.oref_bf16_value.argtypes = [ctypes.c_uint16]
        lib.oref_bf16_value.restype = ctypes.c_double
        lib.oga_calibrate.argtypes = [P, i64, P, P]
        lib.oga_group_mode.argtypes = [P, P, P]
        lib.oga_encode_tile.argtypes = [P, ctypes.c_int, P, P, P]
        lib.oga_decode_tile.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P, P]
        lib.oga_encode_pages.argtypes = [ctypes.c_int, P, i64, P, P, P, P, i32, P, i64, P, u64, P, i32]
        lib.oga_decode_pages.argtypes = [ctypes.c_int, P, i64, P, u64, P, P, i32, P]
        lib.oref_ga_decode_attention.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int, P, P, P, i64, P, u64, P, P,
            i64, P, ctypes.c_int,
        ]
        ci = ctypes.c_int
        lib.of8_value.argtypes = [ci, ctypes.c_uint8]
        lib.of8_value.restype = ctypes.c_double
        lib.of8_from_bf16.argtypes = [ci, ctypes.c_uint16]
        lib.of8_from_bf16.restype = ctypes.c_uint8
        lib.of8_tile_bytes.argtypes = [ci]
        lib.of8_calibrate.argtypes = [ci, P, i64, P, P]
        lib.of8_encode_tile.argtypes = [ci, P, ci, P, P, P]
        lib.of8_decode_tile.argtypes = [ci, P, ci, ci, P, P, P]
        lib.of8_quantize.argtypes = [ci, P, i64, P]
        lib.of8_encode_pages.argtypes = [ci, ci, P, i64, P, P, P, P, i32, P, i64, P, u64, P, i32]
        lib.of8_decode_pages.argtypes = [ci, ci, P, i64, P, u64, P, P, i32, P]
        lib.oref_f8_decode_attention.argtypes = [ci, ci, ci, ci, P, P, ci, P, P, P, i64, P, u64, P, P, i64, P, ci]
        lib.oref_bf16_exponent.argtypes = [ctypes.c_uint16]
        lib.oref_bf16_exponent.restype = ctypes.c_uint
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def block_position(is_v: bool, j: int, lane: int, f: int, i: int) -> tuple[int, int]:
    """(token, dim) in the 16x128 page of storage element (lane, f, i) of block j."""
    tok, dim = ctypes.c_int(), ctypes.c_int()
    _load().oref_block_position(int(is_v), j, lane, f, i, ctypes.byref(tok), ctypes.byref(dim))
    return tok.value, dim.value


def bf16_value(w: int) -> float:
    return _load().oref_bf16_value(int(w) & 0xFFFF)


def bf16_exponent(w: int) -> int:
    return _load().oref_bf16_exponent(int(w) & 0xFFFF)


def encode_block(page: np.ndarray, is_v: bool, j: int) -> tuple[bytes, int]:
    """Encode block j of a [16][128] uint16 page.  Returns (bytes, tag)."""
    page = _c(page, np.uint16).reshape(PAGE, HEAD_DIM)
    out = np.zeros(1024, np.uint8)
    tag = np.zeros(1, np.uint8)
    n = _load().oref_encode_block(_ptr(page), int(is_v), j, _ptr(out), _ptr(tag))
    return out[:n].tobytes(), int(tag[0])


def decode_block(data: bytes, tag: int, is_v: bool, j: int, page: np.ndarray | None = None) -> np.ndarray:
    """Decode one block into (a copy of) a [16][128] uint16 page; returns the page."""
    page = np.zeros((PAGE, HEAD_DIM), np.uint16) if page is None else _c(page, np.uint16).copy()
    buf = np.zeros(1024, np.uint8)
    raw = np.frombuffer(bytes(data), np.uint8)
    buf[: raw.size] = raw
    rc = _load().oref_decode_block(_ptr(buf), tag, int(is_v), j, _ptr(page))
    if rc < 0:
        raise ValueError(f"invalid tag 0x{tag:02x}")
    return page


def encode_pages(raw_pool, src_page, dst_page, dst_seq, meta, arena, cursors, hkv: int) -> int:
    """In-place encode (see oref_encode_pages).  meta: uint64 [P][hkv][2], arena: uint8,
    cursors: uint32 [C][2].  Returns the status bits."""
    raw_pool = _c(raw_pool, np.uint16)
    src, dst, seq = _c(src_page, np.int32), _c(dst_page, np.int32), _c(dst_seq, np.int32)
    for a, dt in ((meta, np.uint64), (arena, np.uint8), (cursors, np.uint32)):
        assert a.dtype == dt and a.flags["C_CONTIGUOUS"]
    num_raw = raw_pool.size // (hkv * 2 * PAGE * HEAD_DIM)
    return _load().oref_encode_pages(
        hkv, _ptr(raw_pool), num_raw, _ptr(src), _ptr(dst), _ptr(seq), src.size, _ptr(meta),
        meta.size // (hkv * 2), _ptr(arena), arena.size, _ptr(cursors), cursors.size // 2,
    )


def decode_pages(meta, arena, pages, hkv: int) -> tuple[np.ndarray, int]:
    """Decode whole pages -> uint16 [n][hkv][2][16][128]; returns (pages, status)."""
    meta = _c(meta, np.uint64)
    arena = _c(arena, np.uint8)
    pages = _c(pages, np.int32)
    out = np.zeros((pages.size, hkv, 2, PAGE, HEAD_DIM), np.uint16)
    st = _load().oref_decode_pages(
        hkv, _ptr(meta), meta.size // (hkv * 2), _ptr(arena), arena.size, _ptr(pages), pages.size, _ptr(out)
    )
    return out, st


def decode_attention(q, page_ids, seq_lens, tail_page, meta, arena, raw_pool, hkv: int, nthreads: int = 1):
    """fp64 attention over compressed pages + raw tail.  q: uint16 [B][Hq][128].
    Returns (out float64 [B][Hq][128], status)."""
    q = _c(q, np.uint16)
    B, hq = q.shape[0], q.shape[1]
    page_ids = _c(page_ids, np.int32).reshape(B, -1)
    seq_lens, tail_page = _c(seq_lens, np.int32), _c(tail_page, np.int32)
    meta, arena, raw_pool = _c(meta, np.uint64), _c(arena, np.uint8), _c(raw_pool, np.uint16)
    out = np.zeros((B, hq, HEAD_DIM), np.float64)
    st = _load().oref_decode_attention(
        hkv, B, hq, _ptr(q), _ptr(page_ids), page_ids.shape[1], _ptr(seq_lens), _ptr(tail_page),
        _ptr(meta), meta.size // (hkv * 2), _ptr(arena), arena.size, _ptr(raw_pool),
        raw_pool.size // (hkv * 2 * PAGE * HEAD_DIM), _ptr(out), nthreads,
    )
    return out, st


def attention_raw(q, page_ids, seq_lens, raw_pool, hkv: int, nthreads: int = 1):
    """fp64 attention over plain BF16 pages.  Returns (out float64 [B][Hq][128], status)."""
    q = _c(q, np.uint16)
    B, hq = q.shape[0], q.shape[1]
    page_ids = _c(page_ids, np.int32).reshape(B, -1)
    seq_lens, raw_pool = _c(seq_lens, np.int32), _c(raw_pool, np.uint16)
    out = np.zeros((B, hq, HEAD_DIM), np.float64)
    st = _load().oref_attention_raw(
        hkv, B, hq, _ptr(q), _ptr(page_ids), page_ids.shape[1], _ptr(seq_lens), _ptr(raw_pool),
        raw_pool.size // (hkv * 2 * PAGE * HEAD_DIM), _ptr(out), nthreads,
    )
    return out, st


# ---------------------------------------------------------------------------------
# group-adaptive additive tiles (oga.c)
# ---------------------------------------------------------------------------------
GA_TILE = 3008  # compressed tile bytes: 2048 sign/fraction + 768 codes + 64 tags + 128 escape slot
GA_RAW = 4096
GA_ENTRY_RAW = 0x80000000
GA_ENTRY_INVALID = 0xFFFFFFFF


def ga_calibrate(pages) -> tuple[np.ndarray, np.ndarray]:
    """Bases of one (layer, head, K|V) from sample pages uint16 [n][16][128] -> (b3, b4),
    each uint8 [128]."""
    pages = _c(pages, np.uint16).reshape(-1, PAGE, HEAD_DIM)
    b3, b4 = np.zeros(HEAD_DIM, np.uint8), np.zeros(HEAD_DIM, np.uint8)
    _load().oga_calibrate(_ptr(pages), pages.shape[0], _ptr(b3), _ptr(b4))
    return b3, b4


def ga_calibrate_pool(raw_pool, pages, hkv: int) -> np.ndarray:
    """Bases of every (head, K|V) of a layer from the listed raw pages -> uint8
    [hkv][2][2][128] (head, K|V, b3|b4, channel)."""
    pool = _c(raw_pool, np.uint16).reshape(-1, hkv, 2, PAGE, HEAD_DIM)
    sel = pool[_c(pages, np.int64)]
    out = np.zeros((hkv, 2, 2, HEAD_DIM), np.uint8)
    for h in range(hkv):
        for kv in range(2):
            out[h, kv, 0], out[h, kv, 1] = ga_calibrate(np.ascontiguousarray(sel[:, h, kv]))
    return out


def ga_group_mode(e, b3, b4) -> int:
    """Mode tag of one group of 8 exponents: 0 (3-bit), 1 (4-bit), 2 (raw)."""
    e, b3, b4 = (_c(x, np.uint32) for x in (e, b3, b4))
    return _load().oga_group_mode(_ptr(e), _ptr(b3), _ptr(b4))


def ga_encode_tile(page, is_v: bool, b3, b4) -> bytes:
    """Encode a [16][128] uint16 page slice -> 3008 (compressed) or 4096 (raw) bytes."""
    page = _c(page, np.uint16).reshape(PAGE, HEAD_DIM)
    b3, b4 = _c(b3, np.uint8), _c(b4, np.uint8)
    out = np.zeros(GA_RAW, np.uint8)
    n = _load().oga_encode_tile(_ptr(page), int(is_v), _ptr(b3), _ptr(b4), _ptr(out))
    return out[:n].tobytes()


def ga_decode_tile(data: bytes, is_v: bool, b3, b4) -> np.ndarray:
    """Decode a tile (its length says which kind) -> uint16 [16][128]."""
    assert len(data) in (GA_TILE, GA_RAW)
    buf = np.frombuffer(bytes(data), np.uint8).copy()
    b3, b4 = _c(b3, np.uint8), _c(b4, np.uint8)
    page = np.zeros((PAGE, HEAD_DIM), np.uint16)
    _load().oga_decode_tile(_ptr(buf), int(len(data) == GA_RAW), int(is_v), _ptr(b3), _ptr(b4), _ptr(page))
    return page


def ga_encode_pages(raw_pool, bases, src_page, dst_page, dst_seq, meta, arena, cursors, hkv: int) -> int:
    """In-place tile encode (see oga_encode_pages).  meta: uint32 [P][hkv][2], arena:
    uint8, cursors: uint32 [C][2] in 64-byte granules.  Returns the status bits."""
    raw_pool, bases = _c(raw_pool, np.uint16), _c(bases, np.uint8)
    src, dst, seq = _c(src_page, np.int32), _c(dst_page, np.int32), _c(dst_seq, np.int32)
    for a, dt in ((meta, np.uint32), (arena, np.uint8), (cursors, np.uint32)):
        assert a.dtype == dt and a.flags["C_CONTIGUOUS"]
    num_raw = raw_pool.size // (hkv * 2 * PAGE * HEAD_DIM)
    return _load().oga_encode_pages(
        hkv, _ptr(raw_pool), num_raw, _ptr(bases), _ptr(src), _ptr(dst), _ptr(seq), src.size, _ptr(meta),
        meta.size // (hkv * 2), _ptr(arena), arena.size, _ptr(cursors), cursors.size // 2,
    )


def ga_decode_pages(meta, arena, bases, pages, hkv: int) -> tuple[np.ndarray, int]:
    """Decode whole pages of tiles -> uint16 [n][hkv][2][16][128]; returns (pages, status)."""
    meta, arena, bases = _c(meta, np.uint32), _c(arena, np.uint8), _c(bases, np.uint8)
    pages = _c(pages, np.int32)
    out = np.zeros((pages.size, hkv, 2, PAGE, HEAD_DIM), np.uint16)
    st = _load().oga_decode_pages(
        hkv, _ptr(meta), meta.size // (hkv * 2), _ptr(arena), arena.size, _ptr(bases), _ptr(pages), pages.size,
        _ptr(out),
    )
    return out, st


def ga_decode_attention(q, page_ids, seq_lens, tail_page, meta, arena, bases, raw_pool, hkv: int,
                        nthreads: int = 1):
    """fp64 attention over group-adaptive tiles + raw tail.  Returns (out, status)."""
    q = _c(q, np.uint16)
    B, hq = q.shape[0], q.shape[1]
    page_ids = _c(page_ids, np.int32).reshape(B, -1)
    seq_lens, tail_page = _c(seq_lens, np.int32), _c(tail_page, np.int32)
    meta, arena, raw_pool = _c(meta, np.uint32), _c(arena, np.uint8), _c(raw_pool, np.uint16)
    bases = _c(bases, np.uint8)
    out = np.zeros((B, hq, HEAD_DIM), np.float64)
    st = _load().oref_ga_decode_attention(
        hkv, B, hq, _ptr(q), _ptr(page_ids), page_ids.shape[1], _ptr(seq_lens), _ptr(tail_page),
        _ptr(meta), meta.size // (hkv * 2), _ptr(arena), arena.size, _ptr(bases), _ptr(raw_pool),
        raw_pool.size // (hkv * 2 * PAGE * HEAD_DIM), _ptr(out), nthreads,
    )
    return out, st


# ---------------------------------------------------------------------------------
# FP8 pages with group-adaptive exponent coding (of8.c)
# ---------------------------------------------------------------------------------
E4M3 = 1
E5M2 = 2
F8_RAW_TILE = 2048


def f8_value(fmt: int, b: int) -> float:
    return _load().of8_value(fmt, int(b) & 0xFF)


def f8_from_bf16(fmt: int, w: int) -> int:
    return int(_load().of8_from_bf16(fmt, int(w) & 0xFFFF))


def f8_quantize(fmt: int, words) -> np.ndarray:
    """BF16 words (uint16 array) -> FP8 bytes of the same shape."""
    a = _c(words, np.uint16)
    out = np.zeros(a.shape, np.uint8)
    _load().of8_quantize(fmt, _ptr(a), a.size, _ptr(out))
    return out


def f8_tile_bytes(fmt: int) -> int:
    return int(_load().of8_tile_bytes(fmt))


def f8_calibrate(fmt: int, pages) -> tuple[np.ndarray, np.ndarray]:
    """Bases from FP8 pages uint8 [n][16][128] of one (head, K|V) -> (b3, b4)."""
    pages = _c(pages, np.uint8).reshape(-1, PAGE, HEAD_DIM)
    b3, b4 = np.zeros(HEAD_DIM, np.uint8), np.zeros(HEAD_DIM, np.uint8)
    _load().of8_calibrate(fmt, _ptr(pages), pages.shape[0], _ptr(b3), _ptr(b4))
    return b3, b4


def f8_calibrate_pool(fmt: int, raw_pool, pages, hkv: int) -> np.ndarray:
    """Bases [hkv][2][2][128] from the FP8 conversion of the listed BF16 raw pages."""
    pool = _c(raw_pool, np.uint16).reshape(-1, hkv, 2, PAGE, HEAD_DIM)
    sel = f8_quantize(fmt, pool[_c(pages, np.int64)])
    out = np.zeros((hkv, 2, 2, HEAD_DIM), np.uint8)
    for h in range(hkv):
        for kv in range(2):
            out[h, kv, 0], out[h, kv, 1] = f8_calibrate(fmt, np.ascontiguousarray(sel[:, h, kv]))
    return out


def f8_encode_tile(fmt: int, page, is_v: bool, b3, b4) -> bytes:
    page = _c(page, np.uint8).reshape(PAGE, HEAD_DIM)
    b3, b4 = _c(b3, np.uint8), _c(b4, np.uint8)
    out = np.zeros(F8_RAW_TILE, np.uint8)
    n = _load().of8_encode_tile(fmt, _ptr(page), int(is_v), _ptr(b3), _ptr(b4), _ptr(out))
    return out[:n].tobytes()


def f8_decode_tile(fmt: int, data: bytes, is_v: bool, b3, b4) -> np.ndarray:
    assert len(data) in (f8_tile_bytes(fmt), F8_RAW_TILE)
    buf = np.frombuffer(bytes(data), np.uint8).copy()
    b3, b4 = _c(b3, np.uint8), _c(b4, np.uint8)
    page = np.zeros((PAGE, HEAD_DIM), np.uint8)
    _load().of8_decode_tile(fmt, _ptr(buf), int(len(data) == F8_RAW_TILE), int(is_v), _ptr(b3), _ptr(b4),
                            _ptr(page))
    return page


def f8_encode_pages(fmt, raw_pool, bases, src_page, dst_page, dst_seq, meta, arena, cursors, hkv: int) -> int:
    raw_pool, bases = _c(raw_pool, np.uint16), _c(bases, np.uint8)
    src, dst, seq = _c(src_page, np.int32), _c(dst_page, np.int32), _c(dst_seq, np.int32)
    for a, dt in ((meta, np.uint32), (arena, np.uint8), (cursors, np.uint32)):
        assert a.dtype == dt and a.flags["C_CONTIGUOUS"]
    num_raw = raw_pool.size // (hkv * 2 * PAGE * HEAD_DIM)
    return _load().of8_encode_pages(
        fmt, hkv, _ptr(raw_pool), num_raw, _ptr(bases), _ptr(src), _ptr(dst), _ptr(seq), src.size, _ptr(meta),
        meta.size // (hkv * 2), _ptr(arena), arena.size, _ptr(cursors), cursors.size // 2,
    )


def f8_decode_pages(fmt, meta, arena, bases, pages, hkv: int) -> tuple[np.ndarray, int]:
    meta, arena, bases = _c(meta, np.uint32), _c(arena, np.uint8), _c(bases, np.uint8)
    pages = _c(pages, np.int32)
    out = np.zeros((pages.size, hkv, 2, PAGE, HEAD_DIM), np.uint8)
    st = _load().of8_decode_pages(fmt, hkv, _ptr(meta), meta.size // (hkv * 2), _ptr(arena), arena.size,
                                  _ptr(bases), _ptr(pages), pages.size, _ptr(out))
    return out, st


def f8_decode_attention(fmt, q, page_ids, seq_lens, tail_page, meta, arena, bases, raw_pool, hkv: int,
                        nthreads: int = 1):
    q = _c(q, np.uint16)
    B, hq = q.shape[0], q.shape[1]
    page_ids = _c(page_ids, np.int32).reshape(B, -1)
    seq_lens, tail_page = _c(seq_lens, np.int32), _c(tail_page, np.int32)
    meta, arena, raw_pool = _c(meta, np.uint32), _c(arena, np.uint8), _c(raw_pool, np.uint16)
    bases = _c(bases, np.uint8)
    out = np.zeros((B, hq, HEAD_DIM), np.float64)
    st = _load().oref_f8_decode_attention(
        fmt, hkv, B, hq, _ptr(q), _ptr(page_ids), page_ids.shape[1], _ptr(seq_lens), _ptr(tail_page),
        _ptr(meta), meta.size // (hkv * 2), _ptr(arena), arena.size, _ptr(bases), _ptr(raw_pool),
        raw_pool.size // (hkv * 2 * PAGE * HEAD_DIM), _ptr(out), nthreads,
    )
    return out, st
