"""Shared set-up for the GPU parity tests: seeded inputs from kvgen, encoded once on
the GPU (libkvz) and once by the CPU oracle, never one from the other."""
from __future__ import annotations

import numpy as np
import torch

import kvgen

# attention tolerance (unit-scale outputs): errors relative to the RMS of the oracle
# output of the run
MAX_REL = 4e-3
MEAN_REL = 5e-4


def check_attention(got: torch.Tensor, ref: np.ndarray, what: str = ""):
    g = got.detach().cpu().double().numpy()
    assert g.shape == ref.shape
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    scale = float(np.sqrt(np.mean(ref ** 2)))
    if scale == 0.0:
        assert np.abs(g).max() == 0.0, what
        return 0.0
    err = np.abs(g - ref)
    assert err.max() <= MAX_REL * scale, f"{what}: max|err| {err.max():.3e} > {MAX_REL} * {scale:.3e}"
    assert err.mean() <= MEAN_REL * scale, f"{what}: mean|err| {err.mean():.3e} > {MEAN_REL} * {scale:.3e}"
    return err.max() / scale


class Layer:
    """One layer of a synthetic workload: raw pool, table, lengths, queries, and the
    compressed form produced by the GPU encoder and, independently, by the oracle."""

    def __init__(self, cfg: kvgen.KVConfig, oracle=None, dev="cuda", seq_lens=None, layer: int = 0,
                 device_gen: bool = False):
        import decode_attention_value_gb300 as kvz

        self.cfg = cfg
        self.kvz = kvz
        hkv = cfg.hkv
        lay = kvgen.gen_layout(cfg)
        self.table = lay["table"]
        self.seq_lens = lay["seq_lens"] if seq_lens is None else torch.as_tensor(seq_lens, dtype=torch.int32)
        gen_dev = dev if device_gen else "cpu"
        pool = kvgen.gen_pages(cfg, cfg.num_pages, layer=layer, device=gen_dev)
        self.g_pool = pool.to(dev)
        self.pool = pool.cpu() if not device_gen else None
        self.q = kvgen.gen_q(cfg, layer=layer)
        self.g_q = self.q.to(dev)
        n_full = (self.seq_lens // kvgen.PAGE).tolist()
        # compressed pages: each sequence's first n_full table entries, cursor = sequence
        src, seq = [], []
        for b in range(cfg.batch):
            src += self.table[b, : n_full[b]].tolist()
            seq += [b] * n_full[b]
        self.src = torch.tensor(src, dtype=torch.int32)
        self.dseq = torch.tensor(seq, dtype=torch.int32)
        self.full = self.table[:, : cfg.full_pages].contiguous()
        tails = []
        for b in range(cfg.batch):
            L = int(self.seq_lens[b])
            tails.append(int(self.table[b, L // 16]) if L % 16 else -1)
        self.tail = torch.tensor(tails, dtype=torch.int32)
        per_seq = (cfg.full_pages + 1) * hkv * 2 * 16  # granules: worst case per sequence
        self.arena_bytes = cfg.batch * per_seq * 256
        self.cursors0 = np.array([[b * per_seq, (b + 1) * per_seq] for b in range(cfg.batch)], np.uint32)
        # GPU encode
        self.meta = torch.zeros((cfg.num_pages, hkv, 2), dtype=torch.int64, device=dev)
        self.arena = torch.zeros(self.arena_bytes, dtype=torch.uint8, device=dev)
        self.cursors = torch.from_numpy(self.cursors0.view(np.int32).copy()).to(dev)
        self.status = kvz.new_status(dev)
        if self.src.numel():
            kvz.encode_pages(self.g_pool, self.src.to(dev), self.src.to(dev), self.dseq.to(dev), self.meta,
                             self.arena, self.cursors, self.status)
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0
        self.o = None
        if oracle is not None and self.pool is not None:
            self.encode_oracle(oracle)

    def encode_oracle(self, oracle):
        cfg = self.cfg
        self.o_pool = kvgen.bits(self.pool)
        self.o_meta = np.zeros((cfg.num_pages, cfg.hkv, 2), np.uint64)
        self.o_arena = np.zeros(self.arena_bytes, np.uint8)
        self.o_cursors = self.cursors0.copy()
        st = oracle.encode_pages(self.o_pool, self.src.numpy(), self.src.numpy(), self.dseq.numpy(), self.o_meta,
                                 self.o_arena, self.o_cursors, cfg.hkv)
        assert st == 0

    def raw_table(self):
        # the raw call's table is one column wider than the compressed one (its tail
        # slot), which gives both calls the same work split
        t = self.table
        if t.shape[1] < self.full.shape[1] + 1:
            pad = torch.full((t.shape[0], self.full.shape[1] + 1 - t.shape[1]), -1, dtype=torch.int32)
            t = torch.cat([t, pad], 1)
        return t.contiguous()

    def workspace(self, raw: bool):
        B, hq, hkv = self.cfg.batch, self.cfg.hq, self.cfg.hkv
        tp = self.raw_table().shape[1] if raw else self.full.shape[1] + 1
        return torch.empty(self.kvz.attention_workspace_size(hkv, B, hq, tp), dtype=torch.uint8, device="cuda")

    def run_compressed(self, out=None, meta=None, status=None, flags=0):
        out = torch.empty((self.cfg.batch, self.cfg.hq, 128), dtype=torch.float32, device="cuda") if out is None else out
        st = self.status if status is None else status
        self.kvz.decode_attention(self.g_q, self.full.cuda(), self.seq_lens.cuda(), self.tail.cuda(),
                                  self.meta if meta is None else meta, self.arena, self.g_pool, out, st,
                                  workspace=self.workspace(False), flags=flags)
        return out

    def run_raw(self, out=None, status=None, flags=0):
        out = torch.empty((self.cfg.batch, self.cfg.hq, 128), dtype=torch.float32, device="cuda") if out is None else out
        st = self.status if status is None else status
        self.kvz.decode_attention_raw(self.g_q, self.raw_table().cuda(), self.seq_lens.cuda(), self.g_pool,
                                      out, st, workspace=self.workspace(True), flags=flags)
        return out

    def oracle_attention(self, oracle, nthreads=8, meta=None):
        return oracle.decode_attention(kvgen.bits(self.q), self.full.numpy(), self.seq_lens.numpy(),
                                       self.tail.numpy(), self.o_meta if meta is None else meta, self.o_arena,
                                       self.o_pool, self.cfg.hkv, nthreads=nthreads)


class GaLayer:
    """The same layer in group-adaptive tiles: bases calibrated on a sample of the
    encoded pages (every second one), tiles encoded by the GPU and, independently, by
    the oracle (each from its own bases)."""

    def __init__(self, base: Layer, oracle=None, sample_step: int = 2):
        kvz, cfg = base.kvz, base.cfg
        self.base, self.kvz, self.cfg = base, kvz, cfg
        hkv = cfg.hkv
        self.sample = base.src[::sample_step].contiguous() if base.src.numel() else torch.zeros(0, dtype=torch.int32)
        per_seq = max(cfg.full_pages, 1) * hkv * 2 * 64  # 64-byte granules: worst case per sequence
        self.arena_bytes = cfg.batch * per_seq * 64
        self.cursors0 = np.array([[b * per_seq, (b + 1) * per_seq] for b in range(cfg.batch)], np.uint32)
        self.bases = torch.zeros((hkv, 2, 2, 128), dtype=torch.uint8, device="cuda")
        self.meta = torch.zeros((cfg.num_pages, hkv, 2), dtype=torch.int32, device="cuda")
        self.arena = torch.zeros(self.arena_bytes, dtype=torch.uint8, device="cuda")
        self.cursors = torch.from_numpy(self.cursors0.view(np.int32).copy()).cuda()
        self.status = kvz.new_status()
        kvz.ga_calibrate(base.g_pool, self.sample.cuda(), self.bases, self.status)
        if base.src.numel():
            s = base.src.cuda()
            kvz.ga_encode_pages(base.g_pool, self.bases, s, s, base.dseq.cuda(), self.meta, self.arena,
                                self.cursors, self.status)
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0
        if oracle is not None and base.pool is not None:
            self.encode_oracle(oracle)

    def encode_oracle(self, oracle):
        cfg, base = self.cfg, self.base
        self.o_pool = kvgen.bits(base.pool)
        self.o_bases = oracle.ga_calibrate_pool(self.o_pool, self.sample.numpy(), cfg.hkv)
        self.o_meta = np.zeros((cfg.num_pages, cfg.hkv, 2), np.uint32)
        self.o_arena = np.zeros(self.arena_bytes, np.uint8)
        self.o_cursors = self.cursors0.copy()
        src = base.src.numpy()
        st = oracle.ga_encode_pages(self.o_pool, self.o_bases, src, src, base.dseq.numpy(), self.o_meta,
                                    self.o_arena, self.o_cursors, cfg.hkv)
        assert st == 0

    def run(self, out=None, meta=None, status=None):
        base = self.base
        out = torch.empty((self.cfg.batch, self.cfg.hq, 128), dtype=torch.float32, device="cuda") if out is None else out
        st = self.status if status is None else status
        self.kvz.ga_decode_attention(base.g_q, base.full.cuda(), base.seq_lens.cuda(), base.tail.cuda(),
                                     self.meta if meta is None else meta, self.arena, self.bases, base.g_pool, out,
                                     st, workspace=base.workspace(False))
        return out

    def oracle_attention(self, oracle, nthreads=8, meta=None):
        base = self.base
        return oracle.ga_decode_attention(kvgen.bits(base.q), base.full.numpy(), base.seq_lens.numpy(),
                                          base.tail.numpy(), self.o_meta if meta is None else meta, self.o_arena,
                                          self.o_bases, self.o_pool, self.cfg.hkv, nthreads=nthreads)


class F8Layer:
    """The same layer with its completed pages converted to FP8 and coded: bases from a
    sample of the encoded pages, tiles encoded by the GPU and, independently, the oracle."""

    def __init__(self, base: Layer, fmt: int, oracle=None, sample_step: int = 2):
        kvz, cfg = base.kvz, base.cfg
        self.base, self.kvz, self.cfg, self.fmt = base, kvz, cfg, fmt
        hkv = cfg.hkv
        self.sample = base.src[::sample_step].contiguous() if base.src.numel() else torch.zeros(0, dtype=torch.int32)
        per_seq = max(cfg.full_pages, 1) * hkv * 2 * 32  # 64-byte granules: worst case (raw 2048 B tiles)
        self.arena_bytes = cfg.batch * per_seq * 64
        self.cursors0 = np.array([[b * per_seq, (b + 1) * per_seq] for b in range(cfg.batch)], np.uint32)
        self.bases = torch.zeros((hkv, 2, 2, 128), dtype=torch.uint8, device="cuda")
        self.meta = torch.zeros((cfg.num_pages, hkv, 2), dtype=torch.int32, device="cuda")
        self.arena = torch.zeros(self.arena_bytes, dtype=torch.uint8, device="cuda")
        self.cursors = torch.from_numpy(self.cursors0.view(np.int32).copy()).cuda()
        self.status = kvz.new_status()
        kvz.f8_calibrate(fmt, base.g_pool, self.sample.cuda(), self.bases, self.status)
        if base.src.numel():
            s = base.src.cuda()
            kvz.f8_encode_pages(fmt, base.g_pool, self.bases, s, s, base.dseq.cuda(), self.meta, self.arena,
                                self.cursors, self.status)
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0
        if oracle is not None and base.pool is not None:
            self.encode_oracle(oracle)

    def encode_oracle(self, oracle):
        cfg, base = self.cfg, self.base
        self.o_pool = kvgen.bits(base.pool)
        self.o_bases = oracle.f8_calibrate_pool(self.fmt, self.o_pool, self.sample.numpy(), cfg.hkv)
        self.o_meta = np.zeros((cfg.num_pages, cfg.hkv, 2), np.uint32)
        self.o_arena = np.zeros(self.arena_bytes, np.uint8)
        self.o_cursors = self.cursors0.copy()
        src = base.src.numpy()
        st = oracle.f8_encode_pages(self.fmt, self.o_pool, self.o_bases, src, src, base.dseq.numpy(), self.o_meta,
                                    self.o_arena, self.o_cursors, cfg.hkv)
        assert st == 0

    def run(self, out=None, meta=None, status=None):
        base = self.base
        out = torch.empty((self.cfg.batch, self.cfg.hq, 128), dtype=torch.float32, device="cuda") if out is None else out
        st = self.status if status is None else status
        self.kvz.f8_decode_attention(self.fmt, base.g_q, base.full.cuda(), base.seq_lens.cuda(), base.tail.cuda(),
                                     self.meta if meta is None else meta, self.arena, self.bases, base.g_pool, out,
                                     st, workspace=base.workspace(False))
        return out

    def oracle_attention(self, oracle, nthreads=8, meta=None):
        base = self.base
        return oracle.f8_decode_attention(self.fmt, kvgen.bits(base.q), base.full.numpy(), base.seq_lens.numpy(),
                                          base.tail.numpy(), self.o_meta if meta is None else meta, self.o_arena,
                                          self.o_bases, self.o_pool, self.cfg.hkv, nthreads=nthreads)
