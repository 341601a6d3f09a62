"""Python binding of libkvz: lossless 12-bit BF16 KV pages, group-adaptive additive
tiles, and paged GQA decode attention over either on one GB300 (sm_103a).

Argument marshalling only: every step runs in the CUDA kernels of ``libkvz.so``
(built in-tree by ``_build.build()``).  Tensors are torch CUDA tensors; the binding
passes their device pointers and the current CUDA stream through the C ABI declared in
``include/kvz.h``.  There is no CPU fallback: importing raises when the library is
missing, and every call raises on a non-zero return code.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

PAGE = 16
HEAD_DIM = 128
GRANULE = 256

STATUS_ARENA_FULL = 1
STATUS_BAD_INDEX = 2
STATUS_BAD_ORDER = 4
STATUS_BAD_META = 8
STATUS_TIMEOUT = 16
STATUS_BAD_TAIL = 32
STATUS_Q_RANGE = 64

ERR_OUT_OF_SPACE = -7

# attention launch flags (kvz_decode_attention_ex / kvz_decode_attention_raw_ex)
ATTN_OVERLAP_PREVIOUS = 1

GA_GRANULE = 64
GA_TILE_BYTES = 3008
GA_RAW_TILE_BYTES = 4096
GA_ENTRY_RAW = 0x80000000
GA_ENTRY_INVALID = 0xFFFFFFFF
F8_E4M3 = 1
F8_E5M2 = 2
F8_TILE_BYTES = {F8_E4M3: 1920, F8_E5M2: 1664}
F8_RAW_TILE_BYTES = 2048

EXPORTS = (
    "kvz_encode_workspace_size", "kvz_encode_pages", "kvz_decode_blocks", "kvz_attention_workspace_size",
    "kvz_decode_attention", "kvz_decode_attention_raw", "kvz_alloc_create", "kvz_alloc_destroy",
    "kvz_alloc_reserve", "kvz_alloc_observe", "kvz_alloc_release", "kvz_alloc_stats",
    "kvz_apply_cursor_updates", "kvz_strerror", "kvz_last_cuda_error", "kvz_device_sm_count",
    "kvz_ga_calibrate", "kvz_ga_encode_pages", "kvz_ga_decode_blocks", "kvz_ga_decode_attention",
    "kvz_selftest_bounded_wait", "kvz_encode_sizes", "kvz_alloc_reserve_granules", "kvz_alloc_room",
    "kvz_f8_calibrate", "kvz_f8_encode_pages", "kvz_f8_decode_blocks", "kvz_f8_decode_attention",
    "kvz_decode_attention_ex", "kvz_decode_attention_raw_ex", "kvz_selftest_late_writer",
)


class KvzError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = _lib.kvz_strerror(code).decode()
        if code == -5:
            msg += f" (cudaError {_lib.kvz_last_cuda_error()})"
        super().__init__(f"{fn} failed: {msg} [{code}]")
        self.code = code


class Dims(ctypes.Structure):
    _fields_ = [("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32)]


def _load() -> ctypes.CDLL:
    if not _build.up_to_date():
        _build.build()  # in-tree nvcc build; raises when the toolkit is missing
    if not os.path.exists(_build.LIB):
        raise ImportError(f"libkvz.so is not built ({_build.LIB})")
    lib = ctypes.CDLL(_build.LIB)
    P, i32, i64, u64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
    sig = {
        "kvz_encode_workspace_size": (sz, [Dims, i32]),
        "kvz_encode_pages": (ctypes.c_int, [Dims, P, i64, P, P, P, i32, P, i64, P, u64, P, i32, P, sz, P, P]),
        "kvz_decode_blocks": (ctypes.c_int, [Dims, P, i64, P, u64, P, i32, P, P, P]),
        "kvz_attention_workspace_size": (sz, [Dims, i32, i32, i32]),
        "kvz_decode_attention": (ctypes.c_int, [Dims, i32, i32, P, P, i32, P, P, P, i64, P, u64, P, i64, P, P, sz, P, P]),
        "kvz_decode_attention_raw": (ctypes.c_int, [Dims, i32, i32, P, P, i32, P, P, i64, P, P, sz, P, P]),
        "kvz_decode_attention_ex": (ctypes.c_int, [Dims, i32, i32, P, P, i32, P, P, P, i64, P, u64, P, i64, P, P, sz,
                                                   P, ctypes.c_uint32, P]),
        "kvz_decode_attention_raw_ex": (ctypes.c_int, [Dims, i32, i32, P, P, i32, P, P, i64, P, P, sz, P,
                                                       ctypes.c_uint32, P]),
        "kvz_selftest_late_writer": (ctypes.c_int, [P, P, u64, u64, P]),
        "kvz_alloc_create": (ctypes.c_int, [u64, ctypes.c_uint32, i32, i32, ctypes.POINTER(P)]),
        "kvz_alloc_destroy": (None, [P]),
        "kvz_alloc_reserve": (ctypes.c_int, [P, P, P, i32, P, P, P, P, P]),
        "kvz_alloc_observe": (ctypes.c_int, [P, u64, P]),
        "kvz_alloc_release": (ctypes.c_int, [P, i32]),
        "kvz_alloc_stats": (ctypes.c_int, [P, P, P, P, P, P]),
        "kvz_apply_cursor_updates": (ctypes.c_int, [P, P, P, i32, P, i32, P]),
        "kvz_ga_calibrate": (ctypes.c_int, [Dims, P, i64, P, i32, P, P, P]),
        "kvz_ga_encode_pages": (ctypes.c_int, [Dims, P, i64, P, P, P, P, i32, P, i64, P, u64, P, i32, P, sz, P, P]),
        "kvz_ga_decode_blocks": (ctypes.c_int, [Dims, P, i64, P, u64, P, P, i32, P, P, P]),
        "kvz_ga_decode_attention": (ctypes.c_int, [Dims, i32, i32, P, P, i32, P, P, P, i64, P, u64, P, P, i64, P, P,
                                                   sz, P, P]),
        "kvz_selftest_bounded_wait": (ctypes.c_int, [u64, P, P, P]),
        "kvz_encode_sizes": (ctypes.c_int, [Dims, P, i64, P, i32, P, P, sz, P, P]),
        "kvz_alloc_reserve_granules": (ctypes.c_int, [P, P, P, i32, P, P, P, P, P]),
        "kvz_alloc_room": (ctypes.c_int, [P, i32, P]),
        "kvz_f8_calibrate": (ctypes.c_int, [Dims, i32, P, i64, P, i32, P, P, P]),
        "kvz_f8_encode_pages": (ctypes.c_int, [Dims, i32, P, i64, P, P, P, P, i32, P, i64, P, u64, P, i32, P, sz, P,
                                               P]),
        "kvz_f8_decode_blocks": (ctypes.c_int, [Dims, i32, P, i64, P, u64, P, P, i32, P, P, P]),
        "kvz_f8_decode_attention": (ctypes.c_int, [Dims, i32, i32, i32, P, P, i32, P, P, P, i64, P, u64, P, P, i64, P,
                                                   P, sz, P, P]),
        "kvz_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "kvz_last_cuda_error": (ctypes.c_int, []),
        "kvz_device_sm_count": (ctypes.c_int, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def lib() -> ctypes.CDLL:
    return _lib


# ------------------------------------------------------------------------------------
# marshalling helpers
# ------------------------------------------------------------------------------------
def _dims(hkv: int) -> Dims:
    return Dims(hkv, HEAD_DIM, PAGE)


def _ptr(t: torch.Tensor | None, dtype=None, name: str = "") -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int | None:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(fn: str, rc: int):
    if rc != 0:
        raise KvzError(fn, rc)


_U64 = (torch.uint64, torch.int64) if hasattr(torch, "uint64") else (torch.int64,)
_U32 = (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ())
_U8 = (torch.uint8,)
_BF16 = (torch.bfloat16, torch.int16)


def _pages_of(pool: torch.Tensor) -> int:
    return pool.numel() // (pool.shape[1] * 2 * PAGE * HEAD_DIM) if pool.numel() else 0


# ------------------------------------------------------------------------------------
# sizes
# ------------------------------------------------------------------------------------
def encode_workspace_size(hkv: int, n: int) -> int:
    return int(_lib.kvz_encode_workspace_size(_dims(hkv), n))


def attention_workspace_size(hkv: int, batch: int, num_q_heads: int, table_pages: int) -> int:
    """Workspace bytes for one attention call; table_pages counts the tail slot
    (compressed: max_pages + 1, raw: max_pages)."""
    size = int(_lib.kvz_attention_workspace_size(_dims(hkv), batch, num_q_heads, table_pages))
    if size == 0:
        raise KvzError("kvz_attention_workspace_size", -1)
    return size


def device_sm_count() -> int:
    return int(_lib.kvz_device_sm_count())


def new_status(device="cuda") -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


# ------------------------------------------------------------------------------------
# the four calls
# ------------------------------------------------------------------------------------
def encode_pages(raw_pool, src_page, dst_page, dst_seq, meta, arena, cursors, status, workspace=None, stream=None):
    """Compress pages raw_pool[src_page[i]] (BF16 [P][Hkv][2][16][128]) into the arena at
    cursors[dst_seq[i]], recording metadata under meta[dst_page[i]] (int64/uint64
    [M][Hkv][2]).  Asynchronous; device-side problems are OR-ed into status."""
    hkv = raw_pool.shape[1]
    n = src_page.numel()
    if workspace is None:
        workspace = torch.empty(encode_workspace_size(hkv, n), dtype=torch.uint8, device=raw_pool.device)
    rc = _lib.kvz_encode_pages(
        _dims(hkv), _ptr(raw_pool, _BF16, "raw_pool"), _pages_of(raw_pool),
        _ptr(src_page, torch.int32, "src_page"), _ptr(dst_page, torch.int32, "dst_page"),
        _ptr(dst_seq, torch.int32, "dst_seq"), n, _ptr(meta, _U64, "meta"), meta.numel() // (hkv * 2),
        _ptr(arena, _U8, "arena"), arena.numel(), _ptr(cursors, _U32, "cursors"), cursors.numel() // 2,
        _ptr(workspace, _U8, "workspace"), workspace.numel(), _ptr(status, _U32, "status"), _stream(stream),
    )
    _check("kvz_encode_pages", rc)


def encode_sizes(raw_pool, src_page, granules, status, workspace=None, stream=None):
    """Granules (int32 [n], device) each page raw_pool[src_page[i]] will take when encoded."""
    hkv = raw_pool.shape[1]
    n = src_page.numel()
    if workspace is None:
        workspace = torch.empty(encode_workspace_size(hkv, n), dtype=torch.uint8, device=raw_pool.device)
    rc = _lib.kvz_encode_sizes(
        _dims(hkv), _ptr(raw_pool, _BF16, "raw_pool"), _pages_of(raw_pool), _ptr(src_page, torch.int32, "src_page"),
        n, _ptr(granules, _U32, "granules"), _ptr(workspace, _U8, "workspace"), workspace.numel(),
        _ptr(status, _U32, "status"), _stream(stream),
    )
    _check("kvz_encode_sizes", rc)


def decode_blocks(meta, arena, pages, out, status, stream=None):
    """Decompress pages (meta page ids) into out: BF16 [n][Hkv][2][16][128]."""
    hkv = out.shape[1]
    rc = _lib.kvz_decode_blocks(
        _dims(hkv), _ptr(meta, _U64, "meta"), meta.numel() // (hkv * 2), _ptr(arena, _U8, "arena"), arena.numel(),
        _ptr(pages, torch.int32, "pages"), pages.numel(), _ptr(out, _BF16, "out"), _ptr(status, _U32, "status"),
        _stream(stream),
    )
    _check("kvz_decode_blocks", rc)


def decode_attention(q, page_ids, seq_lens, tail_page, meta, arena, raw_pool, out, status, workspace=None,
                     stream=None, flags: int = 0):
    """Attention over compressed pages page_ids [B][max_pages] plus raw tail pages;
    q BF16 [B][Hq][128] -> out float32 [B][Hq][128].  flags (ATTN_OVERLAP_PREVIOUS)
    selects kvz_decode_attention_ex."""
    B, hq = q.shape[0], q.shape[1]
    hkv = meta.shape[1] if meta.dim() >= 2 else raw_pool.shape[1]
    max_pages = page_ids.shape[1] if page_ids.dim() == 2 else 0
    if workspace is None:
        workspace = torch.empty(attention_workspace_size(hkv, B, hq, max_pages + 1), dtype=torch.uint8,
                                device=q.device)
    args = (
        _dims(hkv), B, hq, _ptr(q, _BF16, "q"), _ptr(page_ids, torch.int32, "page_ids"), max_pages,
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(tail_page, torch.int32, "tail_page"),
        _ptr(meta, _U64, "meta"), meta.numel() // (hkv * 2), _ptr(arena, _U8, "arena"), arena.numel(),
        _ptr(raw_pool, _BF16, "raw_pool"), _pages_of(raw_pool), _ptr(out, torch.float32, "out"),
        _ptr(workspace, _U8, "workspace"), workspace.numel(), _ptr(status, _U32, "status"),
    )
    if flags:
        _check("kvz_decode_attention_ex", _lib.kvz_decode_attention_ex(*args, int(flags), _stream(stream)))
    else:
        _check("kvz_decode_attention", _lib.kvz_decode_attention(*args, _stream(stream)))


def decode_attention_raw(q, page_ids, seq_lens, raw_pool, out, status, workspace=None, stream=None, flags: int = 0):
    """The same attention over plain BF16 pages page_ids [B][max_pages] (all pages);
    flags (ATTN_OVERLAP_PREVIOUS) selects kvz_decode_attention_raw_ex."""
    B, hq = q.shape[0], q.shape[1]
    hkv = raw_pool.shape[1]
    max_pages = page_ids.shape[1]
    if workspace is None:
        workspace = torch.empty(attention_workspace_size(hkv, B, hq, max_pages), dtype=torch.uint8,
                                device=q.device)
    args = (
        _dims(hkv), B, hq, _ptr(q, _BF16, "q"), _ptr(page_ids, torch.int32, "page_ids"), max_pages,
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(raw_pool, _BF16, "raw_pool"), _pages_of(raw_pool),
        _ptr(out, torch.float32, "out"), _ptr(workspace, _U8, "workspace"), workspace.numel(),
        _ptr(status, _U32, "status"),
    )
    if flags:
        _check("kvz_decode_attention_raw_ex", _lib.kvz_decode_attention_raw_ex(*args, int(flags), _stream(stream)))
    else:
        _check("kvz_decode_attention_raw", _lib.kvz_decode_attention_raw(*args, _stream(stream)))


def apply_cursor_updates(idx, pos, end, cursors, stream=None):
    n = idx.numel()
    rc = _lib.kvz_apply_cursor_updates(
        _ptr(idx, torch.int32, "idx"), _ptr(pos, _U32, "pos"), _ptr(end, _U32, "end"), n,
        _ptr(cursors, _U32, "cursors"), cursors.numel() // 2, _stream(stream),
    )
    _check("kvz_apply_cursor_updates", rc)


# ------------------------------------------------------------------------------------
# group-adaptive additive tiles
# ------------------------------------------------------------------------------------
def ga_calibrate(raw_pool, pages, bases, status, stream=None):
    """Window bases of one layer from the sample pages (int32 raw page ids) into bases:
    uint8 [Hkv][2][2][128]."""
    hkv = raw_pool.shape[1]
    rc = _lib.kvz_ga_calibrate(
        _dims(hkv), _ptr(raw_pool, _BF16, "raw_pool"), _pages_of(raw_pool), _ptr(pages, torch.int32, "pages"),
        pages.numel(), _ptr(bases, _U8, "bases"), _ptr(status, _U32, "status"), _stream(stream),
    )
    _check("kvz_ga_calibrate", rc)


def ga_encode_pages(raw_pool, bases, src_page, dst_page, dst_seq, meta, arena, cursors, status, workspace=None,
                    stream=None):
    """encode_pages for tiles: meta int32/uint32 [M][Hkv][2] entries, cursors in 64-byte
    granules."""
    hkv = raw_pool.shape[1]
    n = src_page.numel()
    if workspace is None:
        workspace = torch.empty(encode_workspace_size(hkv, n), dtype=torch.uint8, device=raw_pool.device)
    rc = _lib.kvz_ga_encode_pages(
        _dims(hkv), _ptr(raw_pool, _BF16, "raw_pool"), _pages_of(raw_pool), _ptr(bases, _U8, "bases"),
        _ptr(src_page, torch.int32, "src_page"), _ptr(dst_page, torch.int32, "dst_page"),
        _ptr(dst_seq, torch.int32, "dst_seq"), n, _ptr(meta, _U32, "meta"), meta.numel() // (hkv * 2),
        _ptr(arena, _U8, "arena"), arena.numel(), _ptr(cursors, _U32, "cursors"), cursors.numel() // 2,
        _ptr(workspace, _U8, "workspace"), workspace.numel(), _ptr(status, _U32, "status"), _stream(stream),
    )
    _check("kvz_ga_encode_pages", rc)


def ga_decode_blocks(meta, arena, bases, pages, out, status, stream=None):
    """Decompress tiles of pages (meta page ids) into out: BF16 [n][Hkv][2][16][128]."""
    hkv = out.shape[1]
    rc = _lib.kvz_ga_decode_blocks(
        _dims(hkv), _ptr(meta, _U32, "meta"), meta.numel() // (hkv * 2), _ptr(arena, _U8, "arena"), arena.numel(),
        _ptr(bases, _U8, "bases"), _ptr(pages, torch.int32, "pages"), pages.numel(), _ptr(out, _BF16, "out"),
        _ptr(status, _U32, "status"), _stream(stream),
    )
    _check("kvz_ga_decode_blocks", rc)


def ga_decode_attention(q, page_ids, seq_lens, tail_page, meta, arena, bases, raw_pool, out, status,
                        workspace=None, stream=None):
    """decode_attention over tiles (meta: int32/uint32 [M][Hkv][2] entries)."""
    B, hq = q.shape[0], q.shape[1]
    hkv = meta.shape[1] if meta.dim() >= 2 else raw_pool.shape[1]
    max_pages = page_ids.shape[1] if page_ids.dim() == 2 else 0
    if workspace is None:
        workspace = torch.empty(attention_workspace_size(hkv, B, hq, max_pages + 1), dtype=torch.uint8,
                                device=q.device)
    rc = _lib.kvz_ga_decode_attention(
        _dims(hkv), B, hq, _ptr(q, _BF16, "q"), _ptr(page_ids, torch.int32, "page_ids"), max_pages,
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(tail_page, torch.int32, "tail_page"),
        _ptr(meta, _U32, "meta"), meta.numel() // (hkv * 2), _ptr(arena, _U8, "arena"), arena.numel(),
        _ptr(bases, _U8, "bases"), _ptr(raw_pool, _BF16, "raw_pool"), _pages_of(raw_pool),
        _ptr(out, torch.float32, "out"), _ptr(workspace, _U8, "workspace"), workspace.numel(),
        _ptr(status, _U32, "status"), _stream(stream),
    )
    _check("kvz_ga_decode_attention", rc)


# ------------------------------------------------------------------------------------
# FP8 tiles (format: F8_E4M3 or F8_E5M2)
# ------------------------------------------------------------------------------------
def f8_calibrate(fmt: int, raw_pool, pages, bases, status, stream=None):
    hkv = raw_pool.shape[1]
    rc = _lib.kvz_f8_calibrate(
        _dims(hkv), fmt, _ptr(raw_pool, _BF16, "raw_pool"), _pages_of(raw_pool), _ptr(pages, torch.int32, "pages"),
        pages.numel(), _ptr(bases, _U8, "bases"), _ptr(status, _U32, "status"), _stream(stream),
    )
    _check("kvz_f8_calibrate", rc)


def f8_encode_pages(fmt: int, raw_pool, bases, src_page, dst_page, dst_seq, meta, arena, cursors, status,
                    workspace=None, stream=None):
    hkv = raw_pool.shape[1]
    n = src_page.numel()
    if workspace is None:
        workspace = torch.empty(encode_workspace_size(hkv, n), dtype=torch.uint8, device=raw_pool.device)
    rc = _lib.kvz_f8_encode_pages(
        _dims(hkv), fmt, _ptr(raw_pool, _BF16, "raw_pool"), _pages_of(raw_pool), _ptr(bases, _U8, "bases"),
        _ptr(src_page, torch.int32, "src_page"), _ptr(dst_page, torch.int32, "dst_page"),
        _ptr(dst_seq, torch.int32, "dst_seq"), n, _ptr(meta, _U32, "meta"), meta.numel() // (hkv * 2),
        _ptr(arena, _U8, "arena"), arena.numel(), _ptr(cursors, _U32, "cursors"), cursors.numel() // 2,
        _ptr(workspace, _U8, "workspace"), workspace.numel(), _ptr(status, _U32, "status"), _stream(stream),
    )
    _check("kvz_f8_encode_pages", rc)


def f8_decode_blocks(fmt: int, meta, arena, bases, pages, out, status, stream=None):
    """Decode to FP8 bytes: out uint8 [n][Hkv][2][16][128]."""
    hkv = out.shape[1]
    rc = _lib.kvz_f8_decode_blocks(
        _dims(hkv), fmt, _ptr(meta, _U32, "meta"), meta.numel() // (hkv * 2), _ptr(arena, _U8, "arena"),
        arena.numel(), _ptr(bases, _U8, "bases"), _ptr(pages, torch.int32, "pages"), pages.numel(),
        _ptr(out, _U8, "out"), _ptr(status, _U32, "status"), _stream(stream),
    )
    _check("kvz_f8_decode_blocks", rc)


def f8_decode_attention(fmt: int, q, page_ids, seq_lens, tail_page, meta, arena, bases, raw_pool, out, status,
                        workspace=None, stream=None):
    B, hq = q.shape[0], q.shape[1]
    hkv = meta.shape[1] if meta.dim() >= 2 else raw_pool.shape[1]
    max_pages = page_ids.shape[1] if page_ids.dim() == 2 else 0
    if workspace is None:
        workspace = torch.empty(attention_workspace_size(hkv, B, hq, max_pages + 1), dtype=torch.uint8,
                                device=q.device)
    rc = _lib.kvz_f8_decode_attention(
        _dims(hkv), fmt, B, hq, _ptr(q, _BF16, "q"), _ptr(page_ids, torch.int32, "page_ids"), max_pages,
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(tail_page, torch.int32, "tail_page"),
        _ptr(meta, _U32, "meta"), meta.numel() // (hkv * 2), _ptr(arena, _U8, "arena"), arena.numel(),
        _ptr(bases, _U8, "bases"), _ptr(raw_pool, _BF16, "raw_pool"), _pages_of(raw_pool),
        _ptr(out, torch.float32, "out"), _ptr(workspace, _U8, "workspace"), workspace.numel(),
        _ptr(status, _U32, "status"), _stream(stream),
    )
    _check("kvz_f8_decode_attention", rc)


def selftest_late_writer(src, dst, delay_ns: int, stream=None):
    """Test helper (kvz_selftest_late_writer): copy src to dst on the device after a delay,
    letting a programmatic dependent launch begin first."""
    if src.numel() * src.element_size() != dst.numel() * dst.element_size():
        raise ValueError("src and dst sizes differ")
    _check("kvz_selftest_late_writer", _lib.kvz_selftest_late_writer(
        _ptr(src, None, "src"), _ptr(dst, None, "dst"), src.numel() * src.element_size(), int(delay_ns),
        _stream(stream)))


def selftest_bounded_wait(limit_ns: int, status, out, stream=None):
    """Device check of the bounded barrier wait (see kvz_selftest_bounded_wait); out:
    int64 [3] on the device."""
    _check("kvz_selftest_bounded_wait", _lib.kvz_selftest_bounded_wait(
        int(limit_ns), _ptr(status, _U32, "status"), _ptr(out, _U64, "out"), _stream(stream)))


# ------------------------------------------------------------------------------------
# host allocator
# ------------------------------------------------------------------------------------
class Allocator:
    """Chunk allocator for the arena (host side of kvz_alloc_*)."""

    def __init__(self, arena_bytes: int, chunk_granules: int, num_cursors: int, num_kv_heads: int):
        h = ctypes.c_void_p()
        _check("kvz_alloc_create", _lib.kvz_alloc_create(arena_bytes, chunk_granules, num_cursors, num_kv_heads,
                                                         ctypes.byref(h)))
        self._h = h
        self.num_cursors = num_cursors

    def __del__(self):
        if getattr(self, "_h", None):
            _lib.kvz_alloc_destroy(self._h)
            self._h = None

    def reserve(self, cursor_ids, pages):
        """Returns (ticket, [(cursor, pos, end), ...]) -- updates to copy to the device."""
        import numpy as np

        ids = np.ascontiguousarray(cursor_ids, dtype=np.int32)
        pg = np.ascontiguousarray(pages, dtype=np.int32)
        n = ids.size
        ui = np.zeros(max(n, 1), np.int32)
        up = np.zeros(max(n, 1), np.uint32)
        ue = np.zeros(max(n, 1), np.uint32)
        nu = ctypes.c_int32()
        tk = ctypes.c_uint64()
        rc = _lib.kvz_alloc_reserve(self._h, ids.ctypes.data, pg.ctypes.data, n, ui.ctypes.data, up.ctypes.data,
                                    ue.ctypes.data, ctypes.byref(nu), ctypes.byref(tk))
        _check("kvz_alloc_reserve", rc)
        k = nu.value
        return tk.value, list(zip(ui[:k].tolist(), up[:k].tolist(), ue[:k].tolist()))

    def reserve_granules(self, cursor_ids, granules):
        """Exact reservation: granules[k] for cursor cursor_ids[k].  Returns (ticket, updates)."""
        import numpy as np

        ids = np.ascontiguousarray(cursor_ids, dtype=np.int32)
        gr = np.ascontiguousarray(granules, dtype=np.uint64)
        n = ids.size
        ui = np.zeros(max(n, 1), np.int32)
        up = np.zeros(max(n, 1), np.uint32)
        ue = np.zeros(max(n, 1), np.uint32)
        nu = ctypes.c_int32()
        tk = ctypes.c_uint64()
        rc = _lib.kvz_alloc_reserve_granules(self._h, ids.ctypes.data, gr.ctypes.data, n, ui.ctypes.data,
                                             up.ctypes.data, ue.ctypes.data, ctypes.byref(nu), ctypes.byref(tk))
        _check("kvz_alloc_reserve_granules", rc)
        k = nu.value
        return tk.value, list(zip(ui[:k].tolist(), up[:k].tolist(), ue[:k].tolist()))

    def room(self, cursor: int) -> int:
        r = ctypes.c_uint64()
        _check("kvz_alloc_room", _lib.kvz_alloc_room(self._h, cursor, ctypes.byref(r)))
        return r.value

    def observe(self, ticket: int, cursors_snapshot):
        import numpy as np

        snap = np.ascontiguousarray(cursors_snapshot, dtype=np.uint32).reshape(-1)
        _check("kvz_alloc_observe", _lib.kvz_alloc_observe(self._h, ticket, snap.ctypes.data))

    def release(self, cursor: int):
        _check("kvz_alloc_release", _lib.kvz_alloc_release(self._h, cursor))

    def stats(self) -> dict:
        held, free, used = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint64()
        ch, cf = ctypes.c_int32(), ctypes.c_int32()
        _check("kvz_alloc_stats", _lib.kvz_alloc_stats(self._h, ctypes.byref(held), ctypes.byref(free),
                                                       ctypes.byref(used), ctypes.byref(ch), ctypes.byref(cf)))
        return {"held_bytes": held.value, "free_bytes": free.value, "used_bytes_bound": used.value,
                "chunks_held": ch.value, "chunks_free": cf.value}
