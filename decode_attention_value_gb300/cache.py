"""Fill-then-finalize paged KV storage over libkvz (GAAC, "Block-Wise Compression
Scheduling"; ZipFusion, the memory-manager paragraph of "How it works").

Host-side bookkeeping only: every byte of KV is written and read by libkvz kernels
(``kvz_encode_pages``, ``kvz_decode_attention``) or by plain tensor copies of token rows.

``CompressedKVCache``: each sequence slot keeps its completed 16-token pages as 12-bit
block groups in one arena shared by all layers and sequences, placed at the slot's device
cursor inside fixed chunks that the host allocator (``kvz_alloc_*``) hands out and takes
back when a sequence is released; the incomplete last page of every layer stays raw BF16
in the slot's tail page until its 16th token arrives, then it is encoded once.

``RawKVCache``: the same interface over plain BF16 pages drawn from a free list of page
slots (the uncompressed baseline of the same budget).
"""
from __future__ import annotations

import numpy as np
import torch

from . import Allocator, ERR_OUT_OF_SPACE, KvzError, PAGE, HEAD_DIM
from . import apply_cursor_updates, attention_workspace_size, decode_attention, decode_attention_raw
from . import encode_pages, encode_sizes, encode_workspace_size, new_status


class OutOfSpace(RuntimeError):
    """The arena has no free chunk for a reservation (nothing was changed)."""


class CompressedKVCache:
    def __init__(self, layers: int, hkv: int, max_seqs: int, max_pages: int, arena_bytes: int,
                 chunk_granules: int = 4096, device="cuda"):
        self.layers, self.hkv, self.max_seqs, self.max_pages = layers, hkv, max_seqs, max_pages
        self.device = torch.device(device)
        dev = self.device
        self.arena = torch.zeros(arena_bytes, dtype=torch.uint8, device=dev)
        # meta page id of slot s's k-th page: s * max_pages + k
        self.meta = torch.zeros((layers, max_seqs * max_pages, hkv, 2), dtype=torch.int64, device=dev)
        # raw tail page of slot s in every layer: raw page id s
        self.tails = torch.zeros((layers, max_seqs, hkv, 2, PAGE, HEAD_DIM), dtype=torch.bfloat16, device=dev)
        self.cursors = torch.zeros((max_seqs, 2), dtype=torch.int32, device=dev)
        self.alloc = Allocator(arena_bytes, chunk_granules, max_seqs, hkv)
        self.chunk_bytes = chunk_granules * 256
        self.max_pages_per_call = max(1, chunk_granules // (32 * hkv))  # one call's worst case fits a chunk
        self.lens = np.zeros(max_seqs, np.int64)
        self.status = new_status(dev)
        self._enc_ws = {}
        self.pages_encoded = 0  # (page, layer) items
        self.granules_encoded = 0  # their exact sizes (256-byte granules)
        self.chunk_grants = 0  # chunks handed to cursors so far (released chunks come back)

    # -- bookkeeping ---------------------------------------------------------------
    def _ws(self, n):
        if n not in self._enc_ws:
            self._enc_ws[n] = torch.empty(encode_workspace_size(self.hkv, n), dtype=torch.uint8, device=self.device)
        return self._enc_ws[n]

    def _reserve(self, slots, granules):
        """Exact reservation (granules per slot, from the encoder's size pass)."""
        try:
            ticket, ups = self.alloc.reserve_granules(slots, granules)
        except KvzError as e:
            if e.code == ERR_OUT_OF_SPACE:
                raise OutOfSpace("no free arena chunk") from None
            raise
        if ups:
            self.chunk_grants += len(ups)
            u = torch.tensor(ups, dtype=torch.int64)
            apply_cursor_updates(u[:, 0].to(torch.int32).to(self.device), u[:, 1].to(torch.int32).to(self.device),
                                 u[:, 2].to(torch.int32).to(self.device), self.cursors)

    def _sizes(self, pools, src):
        """Granules of pages pools[layer][src[i]] in every layer: host int64 [layers][n].
        One size pass over all layers (the layers' pools viewed as one pool)."""
        n, per = src.numel(), pools.shape[1]
        flat = pools.reshape((self.layers * per,) + tuple(pools.shape[2:]))
        ids = (torch.arange(self.layers, dtype=torch.int32, device=self.device)[:, None] * per + src[None]).reshape(-1)
        out = torch.empty(self.layers * n, dtype=torch.int32, device=self.device)
        encode_sizes(flat, ids.contiguous(), out, self.status, workspace=self._ws(self.layers * n))
        return out.cpu().numpy().astype(np.int64).reshape(self.layers, n)

    def stats(self) -> dict:
        return self.alloc.stats()

    def mean_page_layer_bytes(self) -> float:
        """Mean compressed bytes of an encoded (page, layer) so far (None before any)."""
        return self.granules_encoded * 256 / self.pages_encoded if self.pages_encoded else None

    def bytes_per_page_layer(self) -> float:
        """Arena bytes per encoded (page, layer) held by the running sequences, chunk-end
        waste included (None when nothing is held)."""
        used = self.alloc.stats()["used_bytes_bound"]
        held_pages = sum(int(self.lens[s]) // PAGE for s in range(self.max_seqs)) * self.layers
        return used / held_pages if held_pages else None

    # -- lifecycle -----------------------------------------------------------------
    def admit(self, slot: int, prompt: torch.Tensor, n_tokens: int):
        """Prefill-side bulk encode.  prompt: BF16 [layers][ceil(n/16)][hkv][2][16][128],
        the sequence's prompt KV.  Its complete pages are measured (size pass), placed in
        runs that fit the slot's current chunk and then fresh chunks (exact reservations:
        a chunk is left only when the next page does not fit it) and encoded; the partial
        page (if any) becomes the tail.  Raises OutOfSpace when the arena runs out (the
        caller releases the slot)."""
        full, rem = divmod(n_tokens, PAGE)
        if full > self.max_pages:
            raise ValueError("prompt longer than max_pages")
        dev = self.device
        if full:
            src = torch.arange(full, dtype=torch.int32, device=dev)
            dst = (slot * self.max_pages + src).contiguous()
            seq = torch.full((full,), slot, dtype=torch.int32, device=dev)
            sizes = self._sizes(prompt, src)
            chunk = self.chunk_bytes // 256
            if sizes.max() > chunk:
                raise ValueError("a page is larger than a chunk")
            for layer in range(self.layers):
                p = 0
                while p < full:
                    room = self.alloc.room(slot)
                    q, tot = p, 0
                    while q < full and tot + sizes[layer, q] <= room:
                        tot += sizes[layer, q]
                        q += 1
                    if q == p:  # opens a fresh chunk
                        while q < full and tot + sizes[layer, q] <= chunk:
                            tot += sizes[layer, q]
                            q += 1
                    self._reserve([slot], [tot])
                    encode_pages(prompt[layer], src[p:q], dst[p:q], seq[p:q], self.meta[layer], self.arena,
                                 self.cursors, self.status, workspace=self._ws(q - p))
                    p = q
            self.pages_encoded += full * self.layers
            self.granules_encoded += int(sizes.sum())
        if rem:
            self.tails[:, slot] = prompt[:, full]
        self.lens[slot] = n_tokens

    def append(self, slots, kv: torch.Tensor):
        """One new token for each sequence in `slots` (host list, distinct), every layer.
        kv: BF16 [layers][len(slots)][hkv][2][128].  Pages that fill are encoded here.
        Raises OutOfSpace, with nothing changed, when a filled page has no room."""
        slots = list(slots)
        done = sorted(s for s in slots if (self.lens[s] + 1) % PAGE == 0)
        pos = self.lens[slots] % PAGE
        idx = torch.as_tensor(slots, dtype=torch.int64, device=self.device)
        p = torch.as_tensor(pos, dtype=torch.int64, device=self.device)
        saved = self.tails[:, idx].clone() if done else None
        # separated index tensors put the indexed dimension first: [n][layers][hkv][2][128]
        self.tails[:, idx, :, :, p, :] = kv.transpose(0, 1)
        if done:
            try:
                self._finalize(done)
            except OutOfSpace:
                self.tails[:, idx] = saved  # nothing changed
                raise
        self.lens[slots] += 1

    def _finalize(self, done):
        """Encode the filled tail pages of `done` in every layer, placed by exact
        reservation (all-or-nothing check first, so OutOfSpace changes nothing).  All
        layers go through at most two encode calls: first, for every sequence, the layers
        that still fit its current chunk (in layer order); then the rest, each sequence's
        remainder in a fresh chunk.  The layers' tail pages and metadata are viewed as one
        pool and one array, entries ordered by sequence and then layer."""
        dev = self.device
        src = torch.as_tensor(done, dtype=torch.int32, device=dev)
        sizes = self._sizes(self.tails, src)  # [layers][n]
        chunk = self.chunk_bytes // 256
        L, n = self.layers, len(done)
        # per sequence: how many leading layers fit the current chunk's room
        split = []
        for i, s in enumerate(done):
            room, k = self.alloc.room(s), 0
            while k < L and sizes[k, i] <= room:
                room -= sizes[k, i]
                k += 1
            if k < L and int(sizes[k:, i].sum()) > chunk:
                raise ValueError("one page completion of every layer is larger than a chunk")
            split.append(k)
        need = sum(1 for k in split if k < L)
        if need > self.alloc.stats()["chunks_free"]:
            raise OutOfSpace("no free arena chunk")
        pages_per_layer = self.max_seqs * self.max_pages
        pool = self.tails.view((L * self.max_seqs,) + tuple(self.tails.shape[2:]))
        meta = self.meta.view((L * pages_per_layer,) + tuple(self.meta.shape[2:]))
        for phase in range(2):
            seqs, grans, ent_src, ent_dst, ent_seq = [], [], [], [], []
            for i, s in enumerate(done):
                layers = range(split[i]) if phase == 0 else range(split[i], L)
                if not len(layers):
                    continue
                seqs.append(s)
                grans.append(int(sum(sizes[l, i] for l in layers)))
                page = int(self.lens[s]) // PAGE
                for l in layers:
                    ent_src.append(l * self.max_seqs + s)
                    ent_dst.append(l * pages_per_layer + s * self.max_pages + page)
                    ent_seq.append(s)
            if not seqs:
                continue
            self._reserve(seqs, grans)
            t = lambda a: torch.as_tensor(a, dtype=torch.int32, device=dev)
            encode_pages(pool, t(ent_src), t(ent_dst), t(ent_seq), meta, self.arena, self.cursors, self.status,
                         workspace=self._ws(len(ent_src)))
        self.pages_encoded += n * L
        self.granules_encoded += int(sizes.sum())

    def release(self, slot: int):
        self.alloc.release(slot)
        self.lens[slot] = 0

    # -- attention -----------------------------------------------------------------
    def batch_args(self, slots):
        """(page_ids [n][max_pages], seq_lens [n], tail_page [n]) device tensors."""
        slots = np.asarray(list(slots), np.int64)
        lens = self.lens[slots]
        table = slots[:, None] * self.max_pages + np.arange(self.max_pages)[None]
        tail = np.where(lens % PAGE != 0, slots, -1)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(self.device, non_blocking=True)
        return t(table), t(lens), t(tail)

    def workspace(self, batch: int, hq: int):
        return torch.empty(attention_workspace_size(self.hkv, batch, hq, self.max_pages + 1), dtype=torch.uint8,
                           device=self.device)

    def attention(self, layer: int, q, args, out, workspace=None):
        table, lens, tail = args
        decode_attention(q, table, lens, tail, self.meta[layer], self.arena, self.tails[layer], out, self.status,
                         workspace=workspace)


class RawKVCache:
    """Plain BF16 pages from a free list of page slots (shared by all layers)."""

    def __init__(self, layers: int, hkv: int, max_seqs: int, max_pages: int, num_slots: int, device="cuda"):
        self.layers, self.hkv, self.max_seqs, self.max_pages = layers, hkv, max_seqs, max_pages
        self.device = torch.device(device)
        self.pool = torch.zeros((layers, num_slots, hkv, 2, PAGE, HEAD_DIM), dtype=torch.bfloat16, device=self.device)
        self.free = list(range(num_slots - 1, -1, -1))
        self.pages = [[] for _ in range(max_seqs)]
        self.lens = np.zeros(max_seqs, np.int64)
        self.status = new_status(self.device)

    def free_pages(self) -> int:
        return len(self.free)

    def admit(self, slot: int, prompt: torch.Tensor, n_tokens: int):
        n = (n_tokens + PAGE - 1) // PAGE
        if n > len(self.free):
            raise OutOfSpace("no free page slot")
        ids = [self.free.pop() for _ in range(n)]
        self.pages[slot] = ids
        self.lens[slot] = n_tokens
        if n:
            self.pool[:, torch.as_tensor(ids, device=self.device)] = prompt[:, :n]

    def append(self, slots, kv: torch.Tensor):
        slots = list(slots)
        starting = [s for s in slots if self.lens[s] % PAGE == 0]  # a new page starts
        if len(starting) > len(self.free):
            raise OutOfSpace("no free page slot")
        for s in starting:
            self.pages[s].append(self.free.pop())
        page = torch.as_tensor([self.pages[s][int(self.lens[s]) // PAGE] for s in slots], device=self.device)
        pos = torch.as_tensor(self.lens[slots] % PAGE, dtype=torch.int64, device=self.device)
        self.pool[:, page, :, :, pos, :] = kv.transpose(0, 1)
        self.lens[slots] += 1

    def release(self, slot: int):
        self.free.extend(reversed(self.pages[slot]))
        self.pages[slot] = []
        self.lens[slot] = 0

    def batch_args(self, slots):
        slots = list(slots)
        table = np.full((len(slots), self.max_pages + 1), -1, np.int32)
        for r, s in enumerate(slots):
            table[r, : len(self.pages[s])] = self.pages[s]
        lens = self.lens[slots].astype(np.int32)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(self.device, non_blocking=True)
        return t(table), t(lens)

    def workspace(self, batch: int, hq: int):
        return torch.empty(attention_workspace_size(self.hkv, batch, hq, self.max_pages + 1), dtype=torch.uint8,
                           device=self.device)

    def attention(self, layer: int, q, args, out, workspace=None):
        table, lens = args
        decode_attention_raw(q, table, lens, self.pool[layer], out, self.status, workspace=workspace)
