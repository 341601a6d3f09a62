"""Benchmark: paged GQA decode attention over 12-bit compressed BF16 KV pages on GB300.

Default workload: the full Llama-3.1-8B-shaped decode step at 8K context -- 32 layers,
batch 16, 32 query heads, 8 KV heads, head dim 128, 8192 tokens in 512 compressed
16-token pages per sequence (shuffled physical order) plus a raw tail of 1..15 tokens,
each layer with its own seeded KV.  A step is one attention call per layer, in layer
order (attention + split merge, 64 kernel launches): kvz_decode_attention_ex with
KVZ_ATTN_OVERLAP_PREVIOUS, so each layer's start-up overlaps the previous layer's merge
(the same step with plain kvz_decode_attention calls is reported beside it; outputs are
bit-identical).  Every step reads all 32 layers' caches once (14.7 GB compressed, far
more than L2).  Synthetic, seeded inputs (kvgen); the KV is resident in HBM before
timing starts.

Reported: logical-KV GB/s (BF16 K+V bytes attended / time) as `value`, µs per step (the
median of five timed runs of K steps), the in-run raw-BF16 kernel on the same pages, the
compressed-block fraction, the dominant kernel's HBM roofline fraction, an end-to-end
figure through the C ABI with host buffers (every layer's queries in, every layer's
output back, each step), the CPU oracle on the host cores, and as extra keys: one C1
layer (batch 32, 2K context) with encode / standalone decode / decompress-first, one
layer of the 8K stack compressed against raw, the streaming Qwen3-8B-shaped step with
page-completion encodes and the capacity count, one 131072-token layer with the
encode/decode throughput at 1-4 GB, and the full 32-layer 131072-token step.

Timing rules: 10 warm-up steps and 50 timed steps per run by default (at least 3 warm-up
steps whatever the flags); inputs larger than L2 (the stack) or rotating copies
of the KV (single layers: 3 copies, > L2) so every step reads cold data; CUDA events on
the launching stream, synchronize on both sides, max over ranks.  `--impl reference`
times the CPU oracle on the same configuration (the reference arm of this build).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import kvgen  # noqa: E402

METRIC = "decode-attention µs/step & logical KV GB/s; % of HBM roofline; encode GB/s"
OVERLAP = 1  # KVZ_ATTN_OVERLAP_PREVIOUS
FALLBACK_HBM_GBS = 6800.0
RUNS = 5  # timed runs of K steps per measurement; the median is reported


# --------------------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def dist_setup():
    """One process per GPU under torchrun; the GPUs run independent replicas of the
    workload (every (sequence, KV head) unit is independent, nothing is exchanged), so
    the ranks only meet in barriers and in the max-over-ranks timing."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist, rank, ws, local
    return None, rank, ws, local


def max_over_ranks(dist, values, device="cpu"):
    """Element-wise max of per-rank timings (the slowest replica sets the job time)."""
    if dist is None:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_throughput(world: int, bytes_per_rank_step: int, steps: int, ms_total: float) -> float:
    """Whole-job logical GB/s: every rank attends bytes_per_rank_step per step."""
    return world * bytes_per_rank_step * steps / (ms_total * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in ("decode_attention_value_gb300/csrc/attention.cu", "decode_attention_value_gb300/csrc/kvz_device.cuh",
                "decode_attention_value_gb300/csrc/ga.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str = "compressed"):
    """dram bytes per launch of an attention kernel ("compressed" = 12-bit groups,
    "tiles" = group-adaptive tiles) from the committed ncu summary, if it was taken on
    the current kernel source."""
    # the C2 profile is of one layer of the stack: the c2-layer workload's kernel launch
    name = {"c2-layer": "c2"}.get(workload, workload)
    p = os.path.join(ROOT, "profiles", f"k_attn_{kernel}_{name}.md")
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as fh:
        for line in fh:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256_16") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def layer_cfg(name: str) -> kvgen.KVConfig:
    """Single-layer workloads: C1 as it is, one layer of the C2 and C4 stacks."""
    base = {"c1": kvgen.C1, "c2-layer": kvgen.C2, "c4": kvgen.C4}[name]
    return kvgen.KVConfig(**{**base.__dict__, "layers": 1})


def config_dict(workload: str, world: int) -> dict:
    """The `config` object of the JSON line; the same function serves both arms, so the
    GPU line and the reference (oracle) line describe the same workload."""
    par = f"replicas{world}"
    if workload == "c2":
        cfg = kvgen.C2
        return {"workload": cfg.name + "-full-stack", "layers": cfg.layers, "batch": cfg.batch, "q_heads": cfg.hq,
                "kv_heads": cfg.hkv, "head_dim": 128, "page_tokens": 16, "context_tokens": cfg.full_pages * 16,
                "tail_tokens": f"{cfg.tail_min}..{cfg.tail_max}", "page_order": "shuffled",
                "kv": "a separate seeded KV cache per layer", "launch": "overlapped layer calls", "parallelism": par,
                "l2": "inputs larger than L2: each step reads all 32 layers' caches once"}
    if workload == "c3":
        cfg = kvgen.C3
        return {"workload": cfg.name, "layers": cfg.layers, "batch": cfg.batch, "q_heads": cfg.hq,
                "kv_heads": cfg.hkv, "head_dim": 128, "page_tokens": 16, "prompt_tokens": 2048,
                "launch": "overlapped layer calls (layer 0 of a step plain: it follows the appends and encodes)",
                "parallelism": par}
    cfg = layer_cfg(workload)
    return {"workload": cfg.name + ("" if workload == "c1" else "-one-layer"), "layers": 1, "batch": cfg.batch,
            "q_heads": cfg.hq, "kv_heads": cfg.hkv, "head_dim": 128, "page_tokens": 16,
            "context_tokens": cfg.full_pages * 16, "tail_tokens": f"{cfg.tail_min}..{cfg.tail_max}",
            "page_order": "shuffled", "parallelism": par,
            "l2": "inputs larger than L2: 3 rotating KV copies read in turn"}


# --------------------------------------------------------------------------------------
# workload
# --------------------------------------------------------------------------------------
class Workload:
    """One decode layer: raw pool, page table, tails, queries, and `copies` compressed
    copies of the same pages at different addresses (so consecutive steps read cold KV)."""

    def __init__(self, cfg: kvgen.KVConfig, copies: int, layer: int = 0, dev="cuda"):
        import decode_attention_value_gb300 as kvz

        self.kvz, self.cfg = kvz, cfg
        B, hq, hkv = cfg.batch, cfg.hq, cfg.hkv
        lay = kvgen.gen_layout(cfg)
        self.table = lay["table"].to(dev)
        self.seq_lens = lay["seq_lens"].to(dev)
        self.tail_len = lay["tail_len"]
        self.full = self.table[:, : cfg.full_pages].contiguous()
        self.tail = self.table[:, cfg.full_pages].contiguous() if cfg.tail_max > 0 else \
            torch.full((B,), -1, dtype=torch.int32, device=dev)
        self.raw_table = self.table.contiguous() if cfg.tail_max > 0 else \
            torch.cat([self.table, torch.full((B, 1), -1, dtype=torch.int32, device=dev)], 1).contiguous()
        self.q = kvgen.gen_q(cfg, layer=layer, device="cpu").to(dev)
        pool = kvgen.gen_pages(cfg, cfg.num_pages, layer=layer, device=dev)
        self.pools = [pool] + [pool.clone() for _ in range(copies - 1)]
        n = B * cfg.full_pages
        self.src = self.full.reshape(-1).contiguous()
        self.dseq = torch.arange(B, dtype=torch.int32, device=dev).repeat_interleave(cfg.full_pages)
        per = (cfg.full_pages + 1) * hkv * 32
        self.arena_bytes = B * per * 256
        self.cursor0 = torch.tensor([[b * per, (b + 1) * per] for b in range(B)], dtype=torch.int32, device=dev)
        self.metas, self.arenas = [], []
        self.status = kvz.new_status(dev)
        self.enc_ws = torch.empty(kvz.encode_workspace_size(hkv, n), dtype=torch.uint8, device=dev)
        for c in range(copies):
            meta = torch.zeros((cfg.num_pages, hkv, 2), dtype=torch.int64, device=dev)
            arena = torch.zeros(self.arena_bytes, dtype=torch.uint8, device=dev)
            cur = self.cursor0.clone()
            kvz.encode_pages(self.pools[c], self.src, self.src, self.dseq, meta, arena, cur, self.status,
                             workspace=self.enc_ws)
            self.metas.append(meta)
            self.arenas.append(arena)
        self.out = torch.empty((B, hq, 128), dtype=torch.float32, device=dev)
        self.out_raw = torch.empty_like(self.out)
        self.out_df = None
        self.ws_c = torch.empty(kvz.attention_workspace_size(hkv, B, hq, cfg.full_pages + 1), dtype=torch.uint8,
                                device=dev)
        self.ws_r = torch.empty(kvz.attention_workspace_size(hkv, B, hq, self.raw_table.shape[1]),
                                dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        if int(self.status.item()) != 0:
            raise RuntimeError(f"encode status {int(self.status.item())}")
        self.copies = copies
        self._stats()

    def _stats(self):
        cfg = self.cfg
        meta = self.metas[0][self.src.long()]  # [n][hkv][2]
        tags = (meta >> 32) & 0xFFFFFFFF
        raw = torch.zeros_like(tags)
        for j in range(4):
            raw += (((tags >> (8 * j)) & 0xFF) == 0xFF).long()
        nblk = tags.numel() * 4
        self.raw_blocks = int(raw.sum())
        self.blocks = nblk
        self.compressed_fraction = 1.0 - self.raw_blocks / nblk
        self.block_bytes = (nblk - self.raw_blocks) * 768 + self.raw_blocks * 1024
        B, hq, hkv = cfg.batch, cfg.hq, cfg.hkv
        tokens = int(self.seq_lens.sum())
        self.logical_bytes = tokens * hkv * 2 * 128 * 2
        pages_c = B * cfg.full_pages
        tail_bytes = int(self.tail_len.sum()) * hkv * 2 * 128 * 2
        q_bytes = B * hq * 128 * 2
        out_bytes = B * hq * 128 * 4
        # partials: each (unit, CTA) segment writes G x (128 + 2) floats, the merge reads them
        G = hq // hkv
        segs = B * hkv + self.grid_c() - 1
        part_bytes = 2 * segs * G * 130 * 4
        self.alg_bytes_c = (self.block_bytes + pages_c * hkv * 16 + pages_c * hkv * 4 + tail_bytes + q_bytes +
                            out_bytes + part_bytes)
        raw_pages = int(((self.seq_lens + 15) // 16).sum())
        self.alg_bytes_r = (self.logical_bytes + raw_pages * hkv * 4 + q_bytes + out_bytes + part_bytes)
        self.pages_c, self.tail_bytes = pages_c, tail_bytes
        self.bytes_ratio = self.block_bytes / (self.blocks * 1024)

    def grid_c(self):
        # the kernel's grid: (workspace - prefix) / (per-slot bytes) = units + C - 1 slots
        cfg = self.cfg
        pre = ((cfg.batch + 1) * 4 + 15) // 16 * 16
        slots = (self.ws_c.numel() - pre) // (4 * 128 * 4 + 4 * 2 * 4)
        return slots - cfg.batch * cfg.hkv + 1

    def step_c(self, k: int, q=None, out=None, flags: int = 0):
        c = k % self.copies
        kw = {"flags": flags} if flags else {}
        self.kvz.decode_attention(self.q if q is None else q, self.full, self.seq_lens, self.tail, self.metas[c],
                                  self.arenas[c], self.pools[c], self.out if out is None else out, self.status,
                                  workspace=self.ws_c, **kw)

    def setup_decompress_first(self):
        """Scratch BF16 pool for the decompress-first pipeline: the layer's compressed pages
        decoded in table order, then the sequences' raw tail pages."""
        cfg, dev = self.cfg, self.full.device
        B, nf = cfg.batch, cfg.full_pages
        self.df_pool = torch.empty((B * nf + B, cfg.hkv, 2, 16, 128), dtype=torch.bfloat16, device=dev)
        t = torch.arange(B * nf, dtype=torch.int32, device=dev).view(B, nf)
        tail_col = (B * nf + torch.arange(B, dtype=torch.int32, device=dev))[:, None]
        self.df_table = torch.cat([t, tail_col], 1).contiguous()
        self.df_tail_src = self.tail.long().clamp_min(0)
        self.df_ws = torch.empty(self.kvz.attention_workspace_size(cfg.hkv, B, cfg.hq, nf + 1), dtype=torch.uint8,
                                 device=dev)
        self.out_df = torch.empty_like(self.out)

    def step_df_decode(self, k: int):
        """Decompress-first, first half: decode every compressed page of the layer to
        BF16 and put the sequences' tails beside them."""
        c = k % self.copies
        B, nf = self.cfg.batch, self.cfg.full_pages
        self.kvz.decode_blocks(self.metas[c], self.arenas[c], self.src, self.df_pool[: B * nf], self.status)
        self.df_pool[B * nf:] = self.pools[c][self.df_tail_src]

    def step_df_attend(self, k: int):
        """Decompress-first, second half: the raw kernel over the decoded pool."""
        self.kvz.decode_attention_raw(self.q, self.df_table, self.seq_lens, self.df_pool, self.out_df, self.status,
                                      workspace=self.df_ws)

    def step_df(self, k: int):
        self.step_df_decode(k)
        self.step_df_attend(k)

    def step_r(self, k: int, flags: int = 0):
        c = k % self.copies
        kw = {"flags": flags} if flags else {}
        self.kvz.decode_attention_raw(self.q, self.raw_table, self.seq_lens, self.pools[c], self.out_raw,
                                      self.status, workspace=self.ws_r, **kw)


def graph_of(fn, steps: int):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for k in range(steps):
                fn(k)
    torch.cuda.current_stream().wait_stream(s)
    return g


def time_graph(g, reps: int = 1) -> float:
    """ms for `reps` replays of a captured graph, CUDA events on the current stream."""
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(st)
    for _ in range(reps):
        g.replay()
    e1.record(st)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def timed_runs(g, dist=None, runs: int = RUNS) -> list[float]:
    """ms of each of `runs` timed replays of a K-step graph (barrier before each)."""
    out = []
    for _ in range(runs):
        if dist:
            dist.barrier()
        out.append(time_graph(g))
    return out


def runs_summary(ms: list[float], K: int) -> dict:
    us = [m * 1e3 / K for m in ms]
    return {"n": len(us), "us_per_step_median": round(statistics.median(us), 3),
            "us_per_step_mean": round(float(np.mean(us)), 3), "us_per_step_std": round(float(np.std(us)), 3),
            "us_per_step_runs": [round(u, 3) for u in us]}


def soak(g, seconds: float):
    """Replay a graph for a while so the 200 ms clock samples see the GPU under load."""
    until = time.time() + seconds
    while time.time() < until:
        g.replay()
        torch.cuda.synchronize()


def flush_l2(buf: torch.Tensor):
    """Evict L2 by reading a buffer larger than it (a read leaves no dirty lines that a
    timed kernel would then have to write back)."""
    buf.view(torch.int64).sum()


def per_launch_ms(fn, iters: int, flush: torch.Tensor, period: int = 1, prep=None) -> float:
    """Average duration of one call, CUDA events around it, L2 flushed before each call.
    Each call is replayed from a CUDA graph (one per k % period), so the events bracket
    the call's GPU work and not the host's launch overhead; prep(k), if given, runs
    between the flush and the first event (untimed set-up such as a cursor reset)."""
    graphs = [graph_of(lambda _k, p=p: fn(p), 1) for p in range(period)]
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    ts = []
    evs = []
    for k in range(iters):
        flush_l2(flush)
        if prep is not None:
            prep(k)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        graphs[k % period].replay()
        e1.record(st)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    for e0, e1 in evs:
        ts.append(e0.elapsed_time(e1))
    return sum(ts) / len(ts)


# --------------------------------------------------------------------------------------
# CPU oracle (cpu_baseline and the reference arm)
# --------------------------------------------------------------------------------------
def oracle_encode_rate(cfg: kvgen.KVConfig, mib: int = 64, threads: int = 1) -> float:
    """The CPU oracle's encoder (scalar) on `mib` MiB of the workload's pages per thread:
    BF16 GB/s in over all threads (each thread encodes the same pages into its own
    arena; the oracle's C calls release the GIL)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    oracle.build()
    n = max(1, (mib << 20) // (cfg.hkv * 8192))
    pool = kvgen.bits(kvgen.gen_pages(cfg, n))
    src = np.arange(n, dtype=np.int32)
    outs = [(np.zeros((n, cfg.hkv, 2), np.uint64), np.zeros(n * cfg.hkv * 8192, np.uint8)) for _ in range(threads)]

    def work(k):
        meta, arena = outs[k]
        cur = np.array([[0, arena.size // 256]], np.uint32)
        return oracle.encode_pages(pool, src, src, np.zeros(n, np.int32), meta, arena, cur, cfg.hkv)

    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        sts = list(ex.map(work, range(threads)))
    dt = time.perf_counter() - t0
    assert all(st == 0 for st in sts)
    return threads * pool.nbytes / dt / 1e9


class OracleSample:
    """The CPU oracle's decode attention (decode of the compressed pages + fp64 attention)
    on sequences of one layer of the workload: the layer is generated and encoded by the
    oracle once, then timed in passes on all host cores (the oracle's C calls release the
    GIL and thread over (sequence, KV head) units)."""

    def __init__(self, cfg: kvgen.KVConfig, threads: int | None = None):
        import oracle

        oracle.build()
        self.oracle, self.cfg = oracle, cfg
        lay = kvgen.gen_layout(cfg)
        self.table, self.seq_lens = lay["table"].numpy(), lay["seq_lens"].numpy()
        self.pool = kvgen.bits(kvgen.gen_pages(cfg, cfg.num_pages))
        self.q = kvgen.bits(kvgen.gen_q(cfg))
        self.threads = threads or os.cpu_count() or 1
        self.sel, self.prep = None, None

    def _prepare(self, sel):
        cfg = self.cfg
        full = self.table[sel, : cfg.full_pages]
        tail = self.table[sel, cfg.full_pages] if cfg.tail_max > 0 else np.full(len(sel), -1, np.int32)
        meta = np.zeros((cfg.num_pages, cfg.hkv, 2), np.uint64)
        per = (cfg.full_pages + 1) * cfg.hkv * 32
        arena = np.zeros(len(sel) * per * 256, np.uint8)
        cur = np.array([[i * per, (i + 1) * per] for i in range(len(sel))], np.uint32)
        src = full.reshape(-1).astype(np.int32)
        seq = np.repeat(np.arange(len(sel), dtype=np.int32), cfg.full_pages)
        self.oracle.encode_pages(self.pool, src, src, seq, meta, arena, cur, cfg.hkv)
        return full, tail, meta, arena

    def _run(self, sel, prep) -> float:
        full, tail, meta, arena = prep
        t0 = time.perf_counter()
        self.oracle.decode_attention(self.q[sel], full, self.seq_lens[sel], tail, meta, arena, self.pool, self.cfg.hkv,
                                     nthreads=self.threads)
        return time.perf_counter() - t0

    def size_for(self, budget_s: float, seqs_max: int | None = None):
        """Pick as many sequences as one pass of about budget_s seconds takes (calibrated on
        one sequence), encode them once."""
        one = [0]
        t1 = self._run(one, self._prepare(one))
        cfg = self.cfg
        n = max(1, min(seqs_max or cfg.batch, cfg.batch, int(budget_s / max(t1, 1e-6) * min(self.threads, cfg.hkv))))
        self.sel = list(range(n))
        self.prep = self._prepare(self.sel)

    def time(self, budget_s: float):
        """Passes over the chosen sequences until about budget_s seconds have been timed:
        (logical GB/s, seconds timed, sequences per pass, passes, threads)."""
        total, passes = 0.0, 0
        while passes == 0 or (total < budget_s and passes < 1000):
            total += self._run(self.sel, self.prep)
            passes += 1
        logical = int(self.seq_lens[self.sel].sum()) * self.cfg.hkv * 2 * 128 * 2 * passes
        return logical / total / 1e9, total, len(self.sel), passes, self.threads


def oracle_sample(cfg: kvgen.KVConfig, budget_s: float, seqs_max: int | None = None, threads: int | None = None):
    """Time the CPU oracle's decode attention on the workload's sequences for about
    budget_s seconds.  Returns (logical GB/s, seconds timed, sequences per pass, passes,
    threads)."""
    o = OracleSample(cfg, threads)
    o.size_for(budget_s, seqs_max)
    return o.time(budget_s)


# --------------------------------------------------------------------------------------
# measurements
# --------------------------------------------------------------------------------------
def measure_layer(cfg: kvgen.KVConfig, args, dev, local, dist, world: int, rank: int, flush=None,
                  decompress_first: bool = False, codec: bool = False) -> dict:
    """One decode layer, compressed and raw kernels each timed as a graph of K steps over
    rotating KV copies (median of RUNS timed runs).  Optionally the decompress-first
    pipeline (standalone decode into a BF16 scratch pool, then the raw kernel; its two
    legs also timed apart) and the encode / standalone-decode throughput of the layer."""
    import decode_attention_value_gb300 as kvz

    peak, peak_kind = measured_peaks()
    W = Workload(cfg, args.copies, layer=rank, dev=dev)
    for k in range(args.warmup):
        W.step_c(k)
        W.step_r(k)
    torch.cuda.synchronize()
    if int(W.status.item()) != 0:
        raise RuntimeError(f"{cfg.name}: attention status {int(W.status.item())}")
    identical = bool(torch.equal(W.out, W.out_raw))
    K = args.steps
    g_c, g_r = graph_of(W.step_c, K), graph_of(W.step_r, K)
    graphs = {"c": g_c, "r": g_r,
              "co": graph_of(lambda k: W.step_c(k, flags=OVERLAP), K),
              "ro": graph_of(lambda k: W.step_r(k, flags=OVERLAP), K)}
    if decompress_first:
        W.setup_decompress_first()
        graphs["df"] = graph_of(W.step_df, K)
        graphs["dfd"] = graph_of(W.step_df_decode, K)
        graphs["dfa"] = graph_of(W.step_df_attend, K)
    for g in graphs.values():
        g.replay()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        soak(g_c, 0.5)
        ms = {name: timed_runs(g, dist) for name, g in graphs.items()}
        soak(g_c, 0.3)
    clocks = clk.summary()
    med = {name: statistics.median(v) for name, v in ms.items()}
    names = list(med)
    vals = max_over_ranks(dist, [med[n] for n in names], device=dev)
    med = dict(zip(names, vals))
    us_c, us_r = med["c"] * 1e3 / K, med["r"] * 1e3 / K
    achieved = W.alg_bytes_c / (us_c * 1e-6) / 1e9
    achieved_r = W.alg_bytes_r / (us_r * 1e-6) / 1e9
    res = {"workload": cfg.name, "batch": cfg.batch, "context_tokens": cfg.full_pages * 16,
           "us_per_step": round(us_c, 3), "raw_us_per_step": round(us_r, 3),
           "speedup_vs_raw": round(us_r / us_c, 4), "expected_speedup_from_fraction": round(1.0 / W.bytes_ratio, 4),
           "compressed_fraction": round(W.compressed_fraction, 5), "compressed_bytes_ratio": round(W.bytes_ratio, 5),
           "logical_GBps": round(job_throughput(world, W.logical_bytes, K, med["c"]), 2),
           "bit_identical_compressed_vs_raw": identical,
           "roofline": {"achieved": round(achieved, 1), "frac": round(achieved / peak, 4), "peak": peak,
                        "peak_kind": peak_kind, "algorithmic_bytes_per_launch": W.alg_bytes_c},
           "roofline_raw": {"achieved": round(achieved_r, 1), "frac": round(achieved_r / peak, 4),
                            "algorithmic_bytes_per_launch": W.alg_bytes_r},
           "runs": runs_summary(ms["c"], K), "runs_raw": runs_summary(ms["r"], K), "clocks": clocks}
    us_co, us_ro = med["co"] * 1e3 / K, med["ro"] * 1e3 / K
    res["overlapped_launches"] = {
        "us_per_step": round(us_co, 3), "raw_us_per_step": round(us_ro, 3), "speedup_vs_raw": round(us_ro / us_co, 4),
        "logical_GBps": round(job_throughput(world, W.logical_bytes, K, med["co"]), 2),
        "roofline_frac": round(W.alg_bytes_c / (us_co * 1e-6) / 1e9 / peak, 4),
        "how": "each step's call with KVZ_ATTN_OVERLAP_PREVIOUS: its start-up overlaps the previous step's merge"}
    if not torch.equal(W.out, W.out_raw):
        raise RuntimeError(f"{cfg.name}: overlapped calls changed the output")
    if decompress_first:
        if not torch.equal(W.out_df, W.out_raw):
            raise RuntimeError(f"{cfg.name}: decompress-first output differs from the raw kernel's")
        us_df, us_dfd, us_dfa = (med[n] * 1e3 / K for n in ("df", "dfd", "dfa"))
        res["decompress_first"] = {
            "us_per_step": round(us_df, 3), "decode_leg_us": round(us_dfd, 3), "attention_leg_us": round(us_dfa, 3),
            "decode_share": round(us_dfd / (us_dfd + us_dfa), 4), "fused_speedup": round(us_df / us_c, 4),
            "how": "standalone decode of every compressed page into a BF16 scratch pool (plus a copy of the tails), "
                   "then the raw kernel over it; each leg also timed as its own graph"}
    if codec:
        fl = flush if flush is not None else torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        enc_meta = torch.zeros_like(W.metas[0])
        enc_arena = torch.zeros_like(W.arenas[0])
        enc_cur = W.cursor0.clone()

        def enc(k):
            kvz.encode_pages(W.pools[k % W.copies], W.src, W.src, W.dseq, enc_meta, enc_arena, enc_cur, W.status,
                             workspace=W.enc_ws)

        enc_ms = per_launch_ms(enc, 10, fl, period=W.copies, prep=lambda k: enc_cur.copy_(W.cursor0))
        enc_in = W.src.numel() * cfg.hkv * 2 * 16 * 128 * 2
        dec_out = torch.empty((W.src.numel(), cfg.hkv, 2, 16, 128), dtype=torch.bfloat16, device=dev)

        def dec(k):
            kvz.decode_blocks(W.metas[k % W.copies], W.arenas[k % W.copies], W.src, dec_out, W.status)

        dec_ms = per_launch_ms(dec, 10, fl, period=W.copies)
        torch.cuda.synchronize()
        if int(W.status.item()) != 0:
            raise RuntimeError(f"{cfg.name}: codec status {int(W.status.item())}")
        if not torch.equal(dec_out.view(torch.int16), W.pools[(10 - 1) % W.copies][W.src.long()].view(torch.int16)):
            raise RuntimeError(f"{cfg.name}: standalone decode differs from the input pages")
        res["encode_GBps"] = round(enc_in / (enc_ms * 1e-3) / 1e9, 2)
        res["decode_GBps"] = round(enc_in / (dec_ms * 1e-3) / 1e9, 2)
        res["codec_how"] = "one call per graph replay, L2 read-flushed before each; GB/s of BF16 pages in (encode) / out (decode)"
    res["_W"] = W
    return res


def stack_layers(cfg: kvgen.KVConfig, dev) -> list:
    """Every layer of the stack with its own seeded KV, one block table for all layers
    (as a paged KV cache keeps it: each layer has its own pools and metadata behind the
    same page ids) and one attention workspace, the scratch buffer a serving loop hands
    to each layer's call in turn."""
    one = kvgen.KVConfig(**{**cfg.__dict__, "layers": 1})
    layers = [Workload(one, 1, layer=layer, dev=dev) for layer in range(cfg.layers)]
    for W in layers[1:]:
        assert torch.equal(W.table, layers[0].table) and torch.equal(W.seq_lens, layers[0].seq_lens)
        W.table, W.full, W.tail, W.raw_table = layers[0].table, layers[0].full, layers[0].tail, layers[0].raw_table
        W.seq_lens = layers[0].seq_lens
        W.ws_c, W.ws_r = layers[0].ws_c, layers[0].ws_r
    return layers


def stack_e2e(layers, K: int, dev, dist, world: int, flags: int = 0) -> dict:
    """The stack end to end through the C ABI with host buffers.  Per step: one
    host-to-device copy of every layer's queries plus the block table, lengths and tail
    ids (one pinned buffer, back to back, 16-byte aligned), the 32 kvz_decode_attention
    calls, and one device-to-host copy of every layer's fp32 output.  Pipelined as a
    serving engine runs it: a copy stream brings step k+1's inputs in and takes step k's
    outputs back while the neighbouring step computes (device inputs and outputs and the
    pinned outputs double-buffered); the K steps are one CUDA graph.  Also reported: the
    same copies and calls back to back on one stream."""
    kvz = layers[0].kvz
    W0 = layers[0]
    L = len(layers)
    q_all = torch.stack([W.q for W in layers]).contiguous()
    parts = [q_all, W0.full.contiguous(), W0.seq_lens.contiguous(), W0.tail.contiguous()]
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 15) // 16 * 16
    pin_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for t, o in zip(parts, offs):
        nb = t.numel() * t.element_size()
        pin_in[o: o + nb].copy_(t.cpu().contiguous().view(torch.uint8).reshape(-1))
    d_in2 = [torch.empty_like(pin_in, device=dev) for _ in range(2)]
    views2 = [[buf[o: o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(parts, offs)]
              for buf in d_in2]
    out_shape = (L,) + tuple(W0.out.shape)
    out2 = [torch.empty(out_shape, dtype=torch.float32, device=dev) for _ in range(2)]
    pin_out2 = [torch.empty(out_shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    status = kvz.new_status(dev)

    kw = {"flags": flags} if flags else {}

    def calls(views, out):
        q_, t_, l_, tl_ = views
        for i, W in enumerate(layers):
            kvz.decode_attention(q_[i], t_, l_, tl_, W.metas[0], W.arenas[0], W.pools[0], out[i], status,
                                 workspace=W0.ws_c, **kw)

    def serial_step(k):
        d_in2[0].copy_(pin_in, non_blocking=True)
        calls(views2[0], out2[0])
        pin_out2[0].copy_(out2[0], non_blocking=True)

    def pipelined_graph(steps: int):
        s, cs = torch.cuda.Stream(), torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                cs.wait_stream(s)
                ev_in = []
                for k in range(steps + 1):
                    if k < steps:  # inputs of step k (slot k % 2: step k - 2 read it before D2H(k - 2))
                        with torch.cuda.stream(cs):
                            d_in2[k % 2].copy_(pin_in, non_blocking=True)
                            e = torch.cuda.Event()
                            e.record(cs)
                            ev_in.append(e)
                    if k >= 1:  # outputs of step k - 1
                        j = k - 1
                        done = torch.cuda.Event()
                        done.record(s)
                        with torch.cuda.stream(cs):
                            cs.wait_event(done)
                            pin_out2[j % 2].copy_(out2[j % 2], non_blocking=True)
                    if k < steps:
                        s.wait_event(ev_in[k])
                        calls(views2[k % 2], out2[k % 2])
                s.wait_stream(cs)
        torch.cuda.current_stream().wait_stream(s)
        return g

    serial_step(0)
    torch.cuda.synchronize()
    g_ser = graph_of(serial_step, K)
    g_pipe = pipelined_graph(K)
    g_ser.replay()
    g_pipe.replay()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"end-to-end status {int(status.item())}")
    ms_pipe = statistics.median(timed_runs(g_pipe, dist))
    ms_ser = statistics.median(timed_runs(g_ser, dist))
    ms_pipe, ms_ser = max_over_ranks(dist, [ms_pipe, ms_ser], device=dev)
    expect = torch.stack([W.out for W in layers]).cpu()
    for buf in [pin_out2[0], pin_out2[1]]:
        if not torch.equal(buf, expect):
            raise RuntimeError("end-to-end outputs differ from the device outputs")
    logical = sum(W.logical_bytes for W in layers)
    return {"value": round(job_throughput(world, logical, K, ms_pipe), 2), "unit": "GB/s",
            "h2d_bytes_per_step": total, "d2h_bytes_per_step": pin_out2[0].numel() * 4,
            "us_per_step": round(ms_pipe * 1e3 / K, 2),
            "how": "pinned host buffers; per step one host-to-device copy of every layer's queries, the block table, "
                   "lengths and tail ids, the 32 C-ABI calls, one device-to-host copy of every layer's output; the "
                   "copies run on a second stream, overlapping the neighbouring steps (inputs and outputs "
                   "double-buffered); the K steps replayed as one CUDA graph; median of 5 timed runs",
            "serial_value": round(job_throughput(world, logical, K, ms_ser), 2),
            "serial_how": "the same copies and calls issued back to back on one stream",
            "launch": "overlapped (KVZ_ATTN_OVERLAP_PREVIOUS)" if flags else "plain"}


def measure_stack(args, dev, local, dist, world: int, rank: int, cfg: kvgen.KVConfig = kvgen.C2,
                  profile: str = "c2", e2e_leg: bool = True) -> dict:
    """A full decode step over every layer of a stack (the 32-layer 8K step by default),
    compressed and raw, overlapped and plain calls, plus its end-to-end leg."""
    peak, peak_kind = measured_peaks()
    layers = stack_layers(cfg, dev)
    L = cfg.layers
    K = args.steps

    def step_c(k):
        for W in layers:
            W.step_c(0)

    def step_r(k):
        for W in layers:
            W.step_r(0)

    def step_co(k):
        for W in layers:
            W.step_c(0, flags=OVERLAP)

    def step_ro(k):
        for W in layers:
            W.step_r(0, flags=OVERLAP)

    for k in range(args.warmup):
        step_c(k)
        step_r(k)
    torch.cuda.synchronize()
    for W in layers:
        if int(W.status.item()) != 0:
            raise RuntimeError(f"status {int(W.status.item())}")
    identical = all(torch.equal(W.out, W.out_raw) for W in layers)
    ref_out = torch.stack([W.out for W in layers]).clone()
    g_c, g_r = graph_of(step_c, K), graph_of(step_r, K)
    g_co, g_ro = graph_of(step_co, K), graph_of(step_ro, K)
    for g in (g_c, g_r, g_co, g_ro):
        g.replay()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        soak(g_co, 0.6)
        ms_co = timed_runs(g_co, dist)
        ms_ro = timed_runs(g_ro, dist)
        ms_c = timed_runs(g_c, dist)
        ms_r = timed_runs(g_r, dist)
        soak(g_co, 0.3)
    clocks = clk.summary()
    if not (torch.equal(torch.stack([W.out for W in layers]), ref_out)
            and all(torch.equal(W.out, W.out_raw) for W in layers)):
        raise RuntimeError("overlapped calls changed the stack's outputs")
    med_co, med_ro = max_over_ranks(dist, [statistics.median(ms_co), statistics.median(ms_ro)], device=dev)
    med_c, med_r = max_over_ranks(dist, [statistics.median(ms_c), statistics.median(ms_r)], device=dev)
    us_c, us_r = med_c * 1e3 / K, med_r * 1e3 / K  # plain launches
    logical = sum(W.logical_bytes for W in layers)
    alg = sum(W.alg_bytes_c for W in layers)
    alg_r = sum(W.alg_bytes_r for W in layers)
    blocks = sum(W.blocks for W in layers)
    raw_blocks = sum(W.raw_blocks for W in layers)
    block_bytes = sum(W.block_bytes for W in layers)
    e2e = stack_e2e(layers, K, dev, dist, world, flags=OVERLAP) if e2e_leg else None
    us_co, us_ro = med_co * 1e3 / K, med_ro * 1e3 / K
    launch_us = us_co / L  # one attention launch + its merge, averaged over the layers of a step
    achieved = alg / L / (launch_us * 1e-6) / 1e9
    achieved_r = alg_r / (us_ro * 1e-6) / 1e9
    res = {
        "value": round(job_throughput(world, logical, K, med_co), 2), "ms_per_step": round(us_co / 1e3, 5),
        "launch": "overlapped: every layer's call is kvz_decode_attention_ex with KVZ_ATTN_OVERLAP_PREVIOUS, a "
                  "programmatic dependent of the previous layer's merge (outputs bit-identical to plain calls); "
                  "the raw arm the same with kvz_decode_attention_raw_ex",
        "us_per_step": round(us_co, 2), "raw_us_per_step": round(us_ro, 2), "speedup_vs_raw": round(us_ro / us_co, 4),
        "compressed_fraction": round(1 - raw_blocks / blocks, 5),
        "compressed_bytes_ratio": round(block_bytes / (blocks * 1024), 5),
        "expected_speedup_from_fraction": round(blocks * 1024 / block_bytes, 4),
        "bit_identical_compressed_vs_raw": identical,
        "compressed_GB": round(block_bytes / 1e9, 3), "logical_GB_per_step": round(logical / 1e9, 3),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": profiled_traffic(profile), "peak_kind": peak_kind,
                     "kernel": "k_attn<12-bit groups> + k_attn_merge (one layer's call)",
                     "launch_us": round(launch_us, 3), "algorithmic_bytes_per_launch": round(alg / L),
                     "how": f"algorithmic bytes of one layer's call (mean over the {L} layers) / (median step time / "
                            f"{L}); traffic: dram bytes of one launch on one layer of this stack (ncu summary in "
                            "profiles/)"},
        "roofline_raw": {"achieved": round(achieved_r, 1), "frac": round(achieved_r / peak, 4),
                         "algorithmic_bytes_per_step": alg_r},
        "runs": {**runs_summary(ms_co, K), "how": f"{RUNS} timed runs of the {K}-step graph, median reported"},
        "runs_raw": runs_summary(ms_ro, K),
        "clocks": clocks, "gpu_launches": 2 * L * K,
        "plain_launches": {
            "us_per_step": round(us_c, 2), "raw_us_per_step": round(us_r, 2), "speedup_vs_raw": round(us_r / us_c, 4),
            "logical_GBps": round(job_throughput(world, logical, K, med_c), 2),
            "roofline_frac": round(alg / L / (us_c / L * 1e-6) / 1e9 / peak, 4),
            "runs": runs_summary(ms_c, K), "runs_raw": runs_summary(ms_r, K),
            "how": "the same step with kvz_decode_attention / kvz_decode_attention_raw (each layer's call starts "
                   "after the previous one has finished)"},
    }
    if e2e is not None:
        res["e2e"] = e2e
    del layers, g_c, g_r, g_co, g_ro
    torch.cuda.empty_cache()
    return res


def measure_stream(args, dev, local, world: int) -> dict:
    """Streaming decode, Qwen3-8B shape (36 layers, 32/8 heads, batch 64): a 2048-token
    prompt (128 pages per sequence and layer, encoded at prefill), then `decode_steps`
    steps that each append one token per sequence and layer and run attention in every
    layer.  When a sequence's tail page fills (every 16th step) the page is encoded in
    every layer before that step's attention, into chunk slots handed out by the host
    allocator; per-step latency includes the encoding.  The same loop on raw pages gives
    the uncompressed step time.  At the end: sequences that fit in the KV budget."""
    import decode_attention_value_gb300 as kvz

    cfg = kvgen.C3
    B, L, hkv, hq = cfg.batch, cfg.layers, cfg.hkv, cfg.hq
    prompt_pages = cfg.full_pages
    T = args.decode_steps
    dec_pages = (T + 15) // 16
    ppseq = prompt_pages + dec_pages + 1  # raw page slots per sequence: prompt, decode pages, spare
    P = B * ppseq
    # raw pool of every layer; page b*ppseq + k is sequence b's k-th page (meta ids are the same)
    raw = torch.empty((L, P, hkv, 2, 16, 128), dtype=torch.bfloat16, device=dev)
    for layer in range(L):
        raw[layer] = kvgen.gen_pages(cfg, P, layer=layer, device=dev)
    new_kv = kvgen.gen_new_tokens(cfg, T, device=dev)  # [T][L][B][hkv][2][128]
    qs = [kvgen.gen_q(cfg, layer=layer).to(dev) for layer in range(L)]
    ids = torch.arange(B, device=dev, dtype=torch.int32) * ppseq
    table = (ids[:, None] + torch.arange(ppseq - 1, device=dev, dtype=torch.int32)[None]).contiguous()
    full_table = table[:, : prompt_pages + dec_pages].contiguous()
    lens_h = [2048 + t + 1 for t in range(T)]
    seq_lens = torch.tensor([[x] * B for x in lens_h], dtype=torch.int32, device=dev)  # [T][B]
    tails = torch.stack([(ids + prompt_pages + t // 16) if x % 16 else torch.full_like(ids, -1)
                         for t, x in enumerate(lens_h)]).contiguous()
    status = kvz.new_status(dev)
    meta = torch.zeros((L, P, hkv, 2), dtype=torch.int64, device=dev)
    chunk = 32768  # granules (8 MiB)
    worst_seq = L * (prompt_pages + dec_pages) * hkv * 32 * 256
    nchunks = B * (worst_seq // (chunk * 256) + 2)
    arena = torch.zeros(nchunks * chunk * 256, dtype=torch.uint8, device=dev)
    alloc = kvz.Allocator(arena.numel(), chunk, B, hkv)
    cursors = torch.zeros((B, 2), dtype=torch.int32, device=dev)
    enc_ws = torch.empty(kvz.encode_workspace_size(hkv, B * max(16, L)), dtype=torch.uint8, device=dev)
    # every layer's pages as one pool and one metadata array, so a page completion encodes
    # all layers in one call (entries ordered by sequence, then layer: each sequence's
    # groups land in its chunk in layer order, as with one call per layer)
    raw_all = raw.view((L * P,) + tuple(raw.shape[2:]))
    meta_all = meta.view((L * P,) + tuple(meta.shape[2:]))
    lay_off = torch.arange(L, device=dev, dtype=torch.int32) * P
    seqs = np.arange(B, dtype=np.int32)

    def apply(updates):
        if updates:
            u = torch.tensor(updates, dtype=torch.int64)
            kvz.apply_cursor_updates(u[:, 0].to(torch.int32).to(dev), u[:, 1].to(torch.int32).to(dev),
                                     u[:, 2].to(torch.int32).to(dev), cursors)

    # ---- prefill: encode every prompt page of every layer, 16 pages per sequence per call ----
    for k0 in range(0, prompt_pages, 16):
        n = min(16, prompt_pages - k0)
        for layer in range(L):
            ticket, ups = alloc.reserve(seqs, [n] * B)
            apply(ups)
            src = (ids[:, None] + torch.arange(k0, k0 + n, device=dev, dtype=torch.int32)[None]).reshape(-1).contiguous()
            dseq = torch.arange(B, device=dev, dtype=torch.int32).repeat_interleave(n)
            kvz.encode_pages(raw[layer], src, src, dseq, meta[layer], arena, cursors, status, workspace=enc_ws)
            alloc.observe(ticket, cursors.cpu().numpy().view(np.uint32))
    torch.cuda.synchronize()
    assert int(status.item()) == 0, int(status.item())

    out_c = torch.empty((B, hq, 128), dtype=torch.float32, device=dev)
    out_r = torch.empty_like(out_c)
    ws_c = torch.empty(kvz.attention_workspace_size(hkv, B, hq, full_table.shape[1] + 1), dtype=torch.uint8, device=dev)
    ws_r = torch.empty(kvz.attention_workspace_size(hkv, B, hq, table.shape[1]), dtype=torch.uint8, device=dev)
    pin_cur = torch.empty((B, 2), dtype=torch.int32).pin_memory()
    pending = None  # (ticket, event) of the last cursor snapshot in flight

    def append(t):
        j, pos = t // 16, t % 16
        raw[:, (ids + prompt_pages + j).long(), :, :, pos, :] = new_kv[t]

    def step_compressed(t):
        nonlocal pending
        append(t)
        if lens_h[t] % 16 == 0:  # every sequence's tail page just filled: encode it in every layer
            if pending is not None and pending[1].query():
                alloc.observe(pending[0], pin_cur.numpy().view(np.uint32))
                pending = None
            ticket, ups = alloc.reserve(seqs, [L] * B)
            apply(ups)
            page = ids + prompt_pages + t // 16
            src = (page[:, None] + lay_off[None, :]).reshape(-1).contiguous()  # [B][L]
            dseq = torch.arange(B, device=dev, dtype=torch.int32).repeat_interleave(L)
            kvz.encode_pages(raw_all, src, src, dseq, meta_all, arena, cursors, status, workspace=enc_ws)
            pin_cur.copy_(cursors, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record()
            pending = (ticket, ev)
        # layer 0 follows the tail append and the encodes: a plain launch; every later layer
        # follows the previous layer's attention and overlaps its start-up with it
        for layer in range(L):
            kvz.decode_attention(qs[layer], full_table, seq_lens[t], tails[t], meta[layer], arena, raw[layer], out_c,
                                 status, workspace=ws_c, flags=OVERLAP if layer else 0)

    def step_raw(t):
        append(t)
        for layer in range(L):
            kvz.decode_attention_raw(qs[layer], table, seq_lens[t], raw[layer], out_r, status, workspace=ws_r,
                                     flags=OVERLAP if layer else 0)

    def run(step_fn):
        times = []
        for t in range(T):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            step_fn(t)
            torch.cuda.synchronize()
            times.append((time.perf_counter() - t0) * 1e6)
        return times

    # the raw loop re-appends the same tokens at the same places, so both loops see the same KV
    with ClockSampler(local) as clk:
        t_c = run(step_compressed)
        t_r = run(step_raw)
    clocks = clk.summary()
    torch.cuda.synchronize()
    st = int(status.item())
    assert st == 0, st
    identical = bool(torch.equal(out_c, out_r))  # last step: same pages, same split -> same bits
    if pending is not None:
        alloc.observe(pending[0], cursors.cpu().numpy().view(np.uint32))
    stats = alloc.stats()
    enc_steps = [t for t in range(T) if lens_h[t] % 16 == 0]
    plain = [t for t in range(T) if lens_h[t] % 16 != 0]
    meta_per_seq = L * (prompt_pages + dec_pages) * hkv * 16
    used_per_seq = stats["used_bytes_bound"] / B
    held_per_seq = stats["held_bytes"] / B
    raw_per_seq = L * (2048 + T) * hkv * 2 * 128 * 2
    budget = args.budget_gb * 1e9
    logical = [L * B * lens_h[t] * hkv * 512 for t in range(T)]
    med_c = statistics.median(t_c)
    res = {
        "workload": cfg.name, "decode_steps": T, "chunk_bytes": chunk * 256,
        "timing": "wall time per step, synchronised (an engine reading logits every step); median over the steps",
        "logical_GBps": round(world * statistics.mean(logical) / (med_c * 1e-6) / 1e9, 2),
        "us_per_step": round(med_c, 1),
        "us_per_step_mean": round(statistics.mean(t_c), 1),
        "us_per_step_with_encode": round(statistics.median([t_c[t] for t in enc_steps]), 1),
        "us_per_step_without_encode": round(statistics.median([t_c[t] for t in plain]), 1),
        "raw_us_per_step": round(statistics.median(t_r), 1),
        "raw_us_per_step_mean": round(statistics.mean(t_r), 1),
        "speedup_vs_raw": round(statistics.mean(t_r) / statistics.mean(t_c), 4),
        "bit_identical_last_step": identical,
        "capacity": {"budget_bytes": budget, "raw_bytes_per_seq": raw_per_seq,
                     "compressed_bytes_per_seq": round(used_per_seq + meta_per_seq),
                     "compressed_bytes_per_seq_chunk_granular": round(held_per_seq + meta_per_seq),
                     "raw_seqs": int(budget // raw_per_seq),
                     "compressed_seqs": int(budget // (used_per_seq + meta_per_seq)),
                     "compressed_seqs_chunk_granular": int(budget // (held_per_seq + meta_per_seq))},
        "clocks": clocks,
        # attention + merge per layer per step, plus 4 encode launches (prepare, sizes, scan,
        # pack) for all layers at each page completion
        "gpu_launches": T * L * 2 + len(enc_steps) * 4,
    }
    del raw, arena, meta, new_kv
    torch.cuda.empty_cache()
    return res


def codec_sweep(dev, sizes_mb) -> list[dict]:
    """Encode and standalone-decode throughput on `sizes_mb` MB of BF16 pages whose
    per-block exponent spread is uniform in 8..20 (so about 58% of blocks qualify).
    encode GB/s = BF16 bytes in / time; decode GB/s = BF16 bytes out / time."""
    import decode_attention_value_gb300 as kvz

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    hkv = 8
    rows = []
    for mb in sizes_mb:
        pages = mb * (1 << 20) // (hkv * 8192)
        cfg = kvgen.KVConfig(f"spread-sweep-{mb}MB", 1, 1, 32, hkv, pages, spread=(8, 20), seed=40 + mb)
        pool = kvgen.gen_pages(cfg, pages, device=dev)
        src = torch.arange(pages, dtype=torch.int32, device=dev)
        seq = torch.zeros_like(src)
        meta = torch.zeros((pages, hkv, 2), dtype=torch.int64, device=dev)
        arena = torch.zeros(pages * hkv * 8192, dtype=torch.uint8, device=dev)
        cur0 = torch.tensor([[0, arena.numel() // 256]], dtype=torch.int32, device=dev)
        cur = cur0.clone()
        st = kvz.new_status(dev)
        ws = torch.empty(kvz.encode_workspace_size(hkv, pages), dtype=torch.uint8, device=dev)
        out = torch.empty_like(pool)

        def enc(k):
            kvz.encode_pages(pool, src, src, seq, meta, arena, cur, st, workspace=ws)

        def dec(k):
            kvz.decode_blocks(meta, arena, src, out, st)

        cur.copy_(cur0)
        enc(0)
        dec(0)
        torch.cuda.synchronize()
        assert int(st.item()) == 0 and torch.equal(out.view(torch.int16), pool.view(torch.int16))
        reps = 5 if mb <= 1024 else 3
        e_ms = per_launch_ms(enc, reps, flush, prep=lambda k: cur.copy_(cur0))
        d_ms = per_launch_ms(dec, reps, flush)
        nbytes = pool.numel() * 2
        tags = (meta >> 32) & 0xFFFFFFFF
        raw = sum(int((((tags >> (8 * j)) & 0xFF) == 0xFF).sum()) for j in range(4))
        rows.append({"MB": mb, "encode_GBps": round(nbytes / e_ms / 1e6, 1), "decode_GBps": round(nbytes / d_ms / 1e6, 1),
                     "encode_us": round(e_ms * 1e3, 1), "decode_us": round(d_ms * 1e3, 1),
                     "compressed_fraction": round(1 - raw / (tags.numel() * 4), 4)})
        del pool, meta, arena, out, ws
        torch.cuda.empty_cache()
    return rows


def public(d: dict) -> dict:
    """A measurement dict without its private handles."""
    return {k: v for k, v in d.items() if not k.startswith("_")}


class GaCopies:
    """The workload's pages as tiles of one of the tile formats: "ga" (group-adaptive BF16
    tiles), "f8e4" / "f8e5" (pages converted to FP8 E4M3 / E5M2, then coded).  Bases are
    calibrated on the GPU from every 8th encoded page of the layer, then one tile copy is
    encoded per KV copy."""

    def __init__(self, W: Workload, kind: str = "ga", sample_step: int = 8):
        kvz, cfg, dev = W.kvz, W.cfg, W.full.device
        B, hkv = cfg.batch, cfg.hkv
        self.W, self.kind = W, kind
        self.fmt = {"f8e4": kvz.F8_E4M3, "f8e5": kvz.F8_E5M2}.get(kind)
        self.comp_bytes = kvz.GA_TILE_BYTES if kind == "ga" else kvz.F8_TILE_BYTES[self.fmt]
        self.raw_bytes = kvz.GA_RAW_TILE_BYTES if kind == "ga" else kvz.F8_RAW_TILE_BYTES
        self.bases = torch.zeros((hkv, 2, 2, 128), dtype=torch.uint8, device=dev)
        self.sample = W.src[::sample_step].contiguous()
        if kind == "ga":
            kvz.ga_calibrate(W.pools[0], self.sample, self.bases, W.status)
        else:
            kvz.f8_calibrate(self.fmt, W.pools[0], self.sample, self.bases, W.status)
        per = max(cfg.full_pages, 1) * hkv * 2 * (self.raw_bytes // kvz.GA_GRANULE)  # granules: worst case
        self.arena_bytes = B * per * kvz.GA_GRANULE
        self.cursor0 = torch.tensor([[b * per, (b + 1) * per] for b in range(B)], dtype=torch.int32, device=dev)
        self.metas, self.arenas = [], []
        for c in range(W.copies):
            meta = torch.zeros((cfg.num_pages, hkv, 2), dtype=torch.int32, device=dev)
            arena = torch.zeros(self.arena_bytes, dtype=torch.uint8, device=dev)
            self.encode(c, meta, arena, self.cursor0.clone())
            self.metas.append(meta)
            self.arenas.append(arena)
        self.out = torch.empty_like(W.out)
        torch.cuda.synchronize()
        if int(W.status.item()) != 0:
            raise RuntimeError(f"tile encode status {int(W.status.item())}")
        e = self.metas[0][W.src.long()].view(-1)
        raw = ((e.view(torch.int32) < 0) & (e != -1)).sum().item()  # bit 31 set: raw tile
        self.tiles = e.numel()
        self.raw_tiles = int(raw)
        self.tile_bytes = (self.tiles - self.raw_tiles) * self.comp_bytes + self.raw_tiles * self.raw_bytes
        G = cfg.hq // hkv
        segs = B * hkv + W.grid_c() - 1
        part_bytes = 2 * segs * G * 130 * 4
        self.alg_bytes = (self.tile_bytes + W.pages_c * hkv * 8 + W.pages_c * hkv * 4 + hkv * 512 + W.tail_bytes +
                          B * cfg.hq * 128 * 2 + B * cfg.hq * 128 * 4 + part_bytes)

    def encode(self, c, meta, arena, cur):
        W, kvz = self.W, self.W.kvz
        if self.kind == "ga":
            kvz.ga_encode_pages(W.pools[c], self.bases, W.src, W.src, W.dseq, meta, arena, cur, W.status,
                                workspace=W.enc_ws)
        else:
            kvz.f8_encode_pages(self.fmt, W.pools[c], self.bases, W.src, W.src, W.dseq, meta, arena, cur, W.status,
                                workspace=W.enc_ws)

    def decode(self, c, out):
        W, kvz = self.W, self.W.kvz
        if self.kind == "ga":
            kvz.ga_decode_blocks(self.metas[c], self.arenas[c], self.bases, W.src, out, W.status)
        else:
            kvz.f8_decode_blocks(self.fmt, self.metas[c], self.arenas[c], self.bases, W.src, out, W.status)

    def step(self, k: int):
        W = self.W
        c = k % W.copies
        if self.kind == "ga":
            W.kvz.ga_decode_attention(W.q, W.full, W.seq_lens, W.tail, self.metas[c], self.arenas[c], self.bases,
                                      W.pools[c], self.out, W.status, workspace=W.ws_c)
        else:
            W.kvz.f8_decode_attention(self.fmt, W.q, W.full, W.seq_lens, W.tail, self.metas[c], self.arenas[c],
                                      self.bases, W.pools[c], self.out, W.status, workspace=W.ws_c)


def run_ga(args, cfg, dist, rank, world, local):
    """The workload through one of the tile formats (group-adaptive BF16 tiles or FP8
    tiles), timed beside the 12-bit format and the raw kernel on the same pages."""
    torch.cuda.set_device(local)
    import decode_attention_value_gb300 as kvz

    dev = torch.device("cuda", local)
    peak, peak_kind = measured_peaks()
    W = Workload(cfg, args.copies, layer=rank, dev=dev)
    GA = GaCopies(W, args.format)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for k in range(args.warmup):
        GA.step(k)
        W.step_c(k)
        W.step_r(k)
    torch.cuda.synchronize()
    if int(W.status.item()) != 0:
        raise RuntimeError(f"attention status {int(W.status.item())}")
    identical = bool(torch.equal(GA.out, W.out_raw))  # FP8 formats change the values: not expected
    K = args.steps
    g_g, g_c, g_r = graph_of(GA.step, K), graph_of(W.step_c, K), graph_of(W.step_r, K)
    for g in (g_g, g_c, g_r):
        g.replay()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        soak_until = time.time() + 0.6
        while time.time() < soak_until:
            g_g.replay()
            torch.cuda.synchronize()
        if dist:
            dist.barrier()
        ms_g = time_graph(g_g)
        ms_c = time_graph(g_c)
        ms_r = time_graph(g_r)
    clocks = clk.summary()
    ms_g, ms_c, ms_r = max_over_ranks(dist, [ms_g, ms_c, ms_r], device=dev)
    us_g, us_c, us_r = (m * 1e3 / K for m in (ms_g, ms_c, ms_r))
    value = job_throughput(world, W.logical_bytes, K, ms_g)
    achieved = GA.alg_bytes / (us_g * 1e-6) / 1e9
    launch_ms = per_launch_ms(GA.step, max(10, min(K, 40)), flush, period=W.copies)

    enc_meta = torch.zeros_like(GA.metas[0])
    enc_arena = torch.zeros_like(GA.arenas[0])
    enc_cur = GA.cursor0.clone()

    def enc(k):
        GA.encode(k % W.copies, enc_meta, enc_arena, enc_cur)

    enc_ms = per_launch_ms(enc, 10, flush, period=W.copies, prep=lambda k: enc_cur.copy_(GA.cursor0))
    enc_in = W.src.numel() * cfg.hkv * 2 * 16 * 128 * 2
    dec_out = torch.empty((W.src.numel(), cfg.hkv, 2, 16, 128),
                          dtype=torch.bfloat16 if args.format == "ga" else torch.uint8, device=dev)

    def dec(k):
        GA.decode(k % W.copies, dec_out)

    dec_ms = per_launch_ms(dec, 10, flush, period=W.copies)
    torch.cuda.synchronize()
    if int(W.status.item()) != 0:
        raise RuntimeError(f"status {int(W.status.item())}")
    if args.format == "ga" and not torch.equal(dec_out.view(torch.int16),
                                               W.pools[(10 - 1) % W.copies][W.src.long()].view(torch.int16)):
        raise RuntimeError("tile decode differs from the input pages")
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(us_g / 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if args.format == "ga" else args.format.replace("f8", "fp8-"),
        "data": "synthetic",
        "config": {"workload": cfg.name, "format": {"ga": "group-adaptive BF16 tiles", "f8e4": "FP8 E4M3 tiles",
                                                    "f8e5": "FP8 E5M2 tiles"}[args.format],
                   "batch": cfg.batch, "q_heads": cfg.hq,
                   "kv_heads": cfg.hkv, "head_dim": 128, "page_tokens": 16, "context_tokens": cfg.full_pages * 16,
                   "tail_tokens": f"{cfg.tail_min}..{cfg.tail_max}", "page_order": "shuffled",
                   "calibration": "every 8th encoded page of the layer", "parallelism": f"replicas{world}",
                   "l2": f"inputs larger than L2: {args.copies} rotating KV copies"},
        "us_per_step": round(us_g, 3),
        "zf_us_per_step": round(us_c, 3),
        "raw_us_per_step": round(us_r, 3),
        "speedup_vs_raw": round(us_r / us_g, 4),
        "speedup_vs_zf": round(us_c / us_g, 4),
        "tile_bytes_ratio": round(GA.tile_bytes / (GA.tiles * 4096), 5),  # of BF16 bytes
        "raw_tile_fraction": round(GA.raw_tiles / GA.tiles, 5),
        "zf_bytes_ratio": round(W.block_bytes / (W.blocks * 1024), 5),
        "bit_identical_tiles_vs_raw": identical if args.format == "ga" else None,
        "encode_GBps": round(enc_in / (enc_ms * 1e-3) / 1e9, 2),
        "decode_GBps": round(enc_in / (dec_ms * 1e-3) / 1e9, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(args.workload, "tiles") if args.format == "ga" else None,
                     "peak_kind": peak_kind, "kernel": "k_attn<tiles> + k_attn_merge", "launch_us": round(us_g, 3),
                     "cold_single_launch_us": round(launch_ms * 1e3, 3),
                     "algorithmic_bytes_per_launch": GA.alg_bytes},
        "clocks": clocks,
        "gpu_launches": 2 * K,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def run_serve(args, dist, rank, world, local):
    """Toy admission loop over a fixed KV budget (GAAC "Block-Wise Compression
    Scheduling", ZipFusion's memory manager): a FIFO queue of requests (seeded prompt and
    generation lengths) is admitted while the cache reports room for them, each running
    sequence gains one token per step in every layer (pages encoded as they fill,
    attention in every layer), and finished sequences are released so their storage serves
    the next requests.  Run twice on the same requests: compressed pages (12-bit groups in
    recycled arena chunks) and raw pages from a slot free list, both holding the same
    budget.  Reports decode tokens/s, mean and peak concurrency, prefill encode time and
    preemptions."""
    import collections
    import dataclasses

    torch.cuda.set_device(local)
    import decode_attention_value_gb300 as kvz
    from decode_attention_value_gb300.cache import CompressedKVCache, OutOfSpace, RawKVCache

    dev = torch.device("cuda", local)
    L, hkv, hq = 8, 8, 32
    cfg = dataclasses.replace(kvgen.C1, layers=L, seed=77)
    rng = np.random.default_rng(77)
    N = args.serve_requests
    reqs = [(int(rng.integers(512, 2049)), int(rng.integers(64, 257))) for _ in range(N)]
    max_pages = (2048 + 256) // 16 + 1
    max_seqs = 192  # slots (tail pages, meta rows); concurrency stays below
    budget = int(args.serve_budget_gb * 1e9)
    page_layer_raw = hkv * 2 * 16 * 128 * 2  # one page of one layer, BF16
    sig = [kvgen.channel_sigmas(cfg, layer, dev) for layer in range(L)]
    qs = [torch.randn((max_seqs, hq, 128), device=dev).to(torch.bfloat16) for _ in range(L)]
    out = torch.empty((max_seqs, hq, 128), dtype=torch.float32, device=dev)

    def pages_of(r):
        return (r[0] + r[1] + 15) // 16

    def run(kind):
        if kind == "compressed":
            tails_bytes = L * max_seqs * page_layer_raw
            meta_bytes = L * max_seqs * max_pages * hkv * 16
            chunk = 8192  # granules of 256 B = 2 MiB
            arena = (budget - tails_bytes - meta_bytes) // (chunk * 256) * (chunk * 256)
            cache = CompressedKVCache(L, hkv, max_seqs, max_pages, arena, chunk_granules=chunk, device=dev)
        else:
            cache = RawKVCache(L, hkv, max_seqs, max_pages, budget // (L * page_layer_raw), device=dev)
        ws = cache.workspace(max_seqs, hq)
        queue = collections.deque(range(N))
        running = {}  # slot -> [request id, tokens generated]
        free = list(range(max_seqs - 1, -1, -1))
        order = []  # running slots in admission order (newest last)
        gen_rng = torch.Generator(device=dev)
        gen_rng.manual_seed(1234)
        t_decode = t_prefill = t_attn = 0.0
        tokens = steps = preempt = peak = 0
        conc = []

        def worst_left(slot):
            rid, done = running[slot]
            return pages_of(reqs[rid]) - (reqs[rid][0] + done) // 16

        def can_admit(rid):
            if kind == "raw":
                need = pages_of(reqs[rid]) + sum(pages_of(reqs[running[s][0]]) - len(cache.pages[s]) for s in running)
                return cache.free_pages() >= need
            st = cache.stats()
            bpl = (cache.mean_page_layer_bytes() or 32 * hkv * 256) * 1.03  # + chunk-end waste
            committed = sum(worst_left(s) for s in running) * L * bpl
            need = pages_of(reqs[rid]) * L * bpl + cache.chunk_bytes
            return st["free_bytes"] - committed >= need

        while queue or running:
            while queue and free and can_admit(queue[0]):
                rid = queue.popleft()
                slot = free.pop()
                n_tok = reqs[rid][0]
                prompt = torch.stack([kvgen.gen_pages(cfg, (n_tok + 15) // 16, layer=layer, device=dev,
                                                      seed_offset=7919 * rid) for layer in range(L)])
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                try:
                    cache.admit(slot, prompt, n_tok)
                except OutOfSpace:
                    cache.release(slot)
                    free.append(slot)
                    queue.appendleft(rid)
                    break
                torch.cuda.synchronize()
                t_prefill += time.perf_counter() - t0
                running[slot] = [rid, 0]
                order.append(slot)
            if not running:
                raise RuntimeError(f"request {queue[0]} does not fit the budget alone")
            slots = sorted(running)
            x = torch.randn((L, len(slots), hkv, 2, 128), device=dev, generator=gen_rng)
            for layer in range(L):
                x[layer, :, :, 0] *= sig[layer][0]
                x[layer, :, :, 1] *= sig[layer][1]
            kv = x.to(torch.bfloat16)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            while True:
                try:
                    cache.append(slots, kv[:, : len(slots)])
                    break
                except OutOfSpace:  # preempt the newest sequence and retry (its request restarts later)
                    victim = order.pop()
                    cache.release(victim)
                    queue.appendleft(running.pop(victim)[0])
                    free.append(victim)
                    preempt += 1
                    keep = [i for i, s in enumerate(slots) if s != victim]
                    slots = [slots[i] for i in keep]
                    kv = kv[:, keep].contiguous()
            n = len(slots)
            args_b = cache.batch_args(slots)
            q_b = [qs[layer][:n].contiguous() for layer in range(L)]
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for layer in range(L):
                cache.attention(layer, q_b[layer], args_b, out[:n], workspace=ws)
            e1.record()
            torch.cuda.synchronize()
            t_decode += time.perf_counter() - t0
            t_attn += e0.elapsed_time(e1) * 1e-3
            steps += 1
            tokens += n
            conc.append(n)
            peak = max(peak, n)
            for s in slots:
                running[s][1] += 1
                if running[s][1] == reqs[running[s][0]][1]:
                    cache.release(s)
                    del running[s]
                    order.remove(s)
                    free.append(s)
        if int(cache.status.item()) != 0:
            raise RuntimeError(f"{kind}: status {int(cache.status.item())}")
        res = {"decode_tokens_per_s": round(tokens / t_decode, 1), "steps": steps, "tokens": tokens,
               "mean_concurrency": round(statistics.mean(conc), 2), "peak_concurrency": peak,
               "decode_s": round(t_decode, 3), "attention_s": round(t_attn, 4),
               "attention_us_per_step": round(t_attn * 1e6 / steps, 1),
               "attention_us_per_token": round(t_attn * 1e6 / tokens, 3),
               "prefill_encode_s": round(t_prefill, 3), "preemptions": preempt}
        if kind == "compressed":
            res["arena_bytes"] = cache.arena.numel()
            res["mean_page_layer_bytes"] = round(cache.mean_page_layer_bytes(), 1)
            res["raw_page_layer_bytes"] = page_layer_raw
            res["chunk_grants"] = cache.chunk_grants
            res["arena_chunks"] = cache.arena.numel() // cache.chunk_bytes
        return res

    with ClockSampler(local) as clk:
        comp = run("compressed")
        raw = run("raw")
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": comp["decode_tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
        "steps": comp["steps"], "warmup": 0, "ms_per_step": round(comp["decode_s"] * 1e3 / comp["steps"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "toy admission loop", "layers": L, "q_heads": hq, "kv_heads": hkv, "head_dim": 128,
                   "requests": N, "prompt_tokens": "512..2048", "generated_tokens": "64..256",
                   "kv_budget_bytes": budget, "timing": "wall time of decode steps (append + encodes + attention in "
                   "every layer), synchronised; prefill encodes timed apart"},
        "compressed": comp, "raw": raw,
        "speedup_vs_raw": round(comp["decode_tokens_per_s"] / raw["decode_tokens_per_s"], 4),
        "attention_speedup_per_token_vs_raw": round(raw["attention_us_per_token"] / comp["attention_us_per_token"], 4),
        "concurrency_gain_vs_raw": round(comp["mean_concurrency"] / raw["mean_concurrency"], 4),
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def run_spread_sweep(args, dist, rank, local):
    """The C4 shape (B=2, 8192 full pages + tail, 32/8 heads) with every block's exponent
    spread fixed at S = 8..20, which moves the compressed fraction from 1 to 0 (eligible
    iff S <= 14, or S = 15 with an even lowest exponent).  Per S: compressed fraction,
    bytes ratio, µs per step compressed and raw (graph replays over 3 rotating copies)."""
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rows = []
    for S in range(8, 21):
        cfg = kvgen.KVConfig(f"long-ctx-spread{S}", 1, 2, 32, 8, 8192, tail_min=1, tail_max=15, spread=(S, S),
                             seed=400 + S)
        W = Workload(cfg, 3, dev=dev)
        for k in range(3):
            W.step_c(k)
            W.step_r(k)
        torch.cuda.synchronize()
        if int(W.status.item()) != 0 or not torch.equal(W.out, W.out_raw):
            raise RuntimeError(f"S={S}: status {int(W.status.item())} or outputs differ")
        K = max(10, min(args.steps, 30))
        g_c, g_r = graph_of(W.step_c, K), graph_of(W.step_r, K)
        g_c.replay()
        g_r.replay()
        ms_c, ms_r = time_graph(g_c), time_graph(g_r)
        ms_c, ms_r = max_over_ranks(dist, [ms_c, ms_r], device=dev)
        ratio = W.block_bytes / (W.blocks * 1024)
        rows.append({"spread": S, "compressed_fraction": round(W.compressed_fraction, 4),
                     "bytes_ratio": round(ratio, 4), "us_compressed": round(ms_c * 1e3 / K, 2),
                     "us_raw": round(ms_r * 1e3 / K, 2), "speedup": round(ms_r / ms_c, 4),
                     "byte_speedup_bound": round(1.0 / ratio, 4)})
        del W, g_c, g_r
        torch.cuda.empty_cache()
    if rank == 0:
        print(json.dumps({"metric": "attention µs/step vs compressed fraction (fixed exponent spread)",
                          "config": {"batch": 2, "context_tokens": 131072, "q_heads": 32, "kv_heads": 8,
                                     "tail_tokens": "1..15"}, "rows": rows, "data": "synthetic"}), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def cpu_baseline_line(cfg: kvgen.KVConfig, budget: float, step_logical: int, layers: int = 1) -> dict:
    """The oracle (decode of compressed pages + fp64 attention) on the host cores, on a
    bounded sample of one layer of the workload, with one-core and encoder figures."""
    gbps, secs, nseq, passes, threads = oracle_sample(cfg, budget)
    cpu = {"value": round(gbps, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
           "us_per_step": round(step_logical / (gbps * 1e9) * 1e6, 1),
           "sample": f"{nseq} of {cfg.batch} sequences x {cfg.hkv} KV heads of one layer (decode of compressed pages "
                     f"+ fp64 attention), {passes} passes, {secs:.1f} s"
                     + (f"; us_per_step scales the rate to the {layers}-layer step" if layers > 1 else "")}
    g1, s1, n1, p1, _ = oracle_sample(cfg, min(4.0, budget / 3), threads=1)
    cpu["extra"] = {"attention_1core_GBps": round(g1, 3),
                    "attention_1core_sample": f"{n1} sequences, {p1} passes, {s1:.1f} s",
                    "encode_1core_GBps": round(oracle_encode_rate(cfg), 3),
                    "encode_sample": "64 MiB of the layer's pages, scalar oracle encoder, one thread",
                    "encode_allcores_GBps": round(oracle_encode_rate(cfg, 32, threads), 3),
                    "encode_allcores_sample": f"{threads} threads x 32 MiB of the layer's pages"}
    return cpu


def base_line(workload: str, world: int, args, value: float, us_step: float) -> dict:
    return {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(us_step / 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_dict(workload, world)}


def run_default(args, dist, rank, world, local):
    """Headline: the full 32-layer 8K decode step (C2).  Extra keys: one C1 layer, one
    layer of the 8K stack, one 131072-token layer with the codec throughput at 1-4 GB,
    the streaming C3 step with page-completion encodes and the capacity count, and the
    full 32-layer 131072-token step (C4)."""
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    S = measure_stack(args, dev, local, dist, world, rank)
    extras = {}
    if not args.no_extras:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        for key, wl, df, codec in (("at_8k_context", "c2-layer", True, True), ("c1_layer", "c1", True, True),
                                   ("c4_layer", "c4", False, False)):
            r = measure_layer(layer_cfg(wl), args, dev, local, dist, world, rank, flush, decompress_first=df,
                              codec=codec)
            r["roofline"]["traffic"] = profiled_traffic(wl)
            del r["_W"]
            torch.cuda.empty_cache()
            extras[key] = public(r)
        rows = codec_sweep(dev, [1024, 4096])
        extras["c4_layer"]["codec_sweep"] = rows
        extras["c4_layer"]["encode_GBps_max"] = max(r["encode_GBps"] for r in rows)
        extras["c4_layer"]["decode_GBps_max"] = max(r["decode_GBps"] for r in rows)
        del flush
        torch.cuda.empty_cache()
        extras["c3_streaming"] = measure_stream(args, dev, local, world)
        # the 131072-token stack: every layer's call of one decode step (32 x ~0.92 GB compressed)
        S4 = measure_stack(args, dev, local, dist, world, rank, cfg=kvgen.C4, profile="c4", e2e_leg=False)
        extras["c4_stack"] = {"workload": kvgen.C4.name + "-full-stack", "layers": kvgen.C4.layers,
                              "batch": kvgen.C4.batch, "context_tokens": kvgen.C4.full_pages * 16,
                              "logical_GBps": S4["value"],
                              **{k: v for k, v in S4.items() if k not in ("value", "ms_per_step", "launch")}}
    cpu = None
    cfg1 = kvgen.KVConfig(**{**kvgen.C2.__dict__, "layers": 1})
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_line(cfg1, args.cpu_budget, int(S["logical_GB_per_step"] * 1e9), kvgen.C2.layers)
    line = base_line("c2", world, args, S["value"], S["us_per_step"])
    line.update({k: v for k, v in S.items() if k not in ("value", "ms_per_step")})
    if "at_8k_context" in extras:
        line["encode_GBps"] = extras["at_8k_context"]["encode_GBps"]
        line["decode_GBps"] = extras["at_8k_context"]["decode_GBps"]
        line["codec_note"] = "encode / standalone decode of one layer of this stack (BF16 GB/s in / out)"
    line["cpu_baseline"] = cpu
    line.update(extras)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def run_layer(args, dist, rank, world, local):
    """One layer (C1, one layer of C2, or one C4 layer) as the headline."""
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = layer_cfg(args.workload)
    r = measure_layer(cfg, args, dev, local, dist, world, rank, decompress_first=True, codec=True)
    W = r.pop("_W")
    e2e = stack_e2e([W], args.steps, dev, dist, world)
    line = base_line(args.workload, world, args, r["logical_GBps"], r["us_per_step"])
    roof = r.pop("roofline")
    line["roofline"] = {"bound": "hbm", "achieved": roof["achieved"], "peak": roof["peak"], "unit": "GB/s",
                        "frac": roof["frac"], "traffic": profiled_traffic(args.workload),
                        "peak_kind": roof["peak_kind"], "kernel": "k_attn<12-bit groups> + k_attn_merge",
                        "launch_us": r["us_per_step"],
                        "algorithmic_bytes_per_launch": roof["algorithmic_bytes_per_launch"]}
    line.update({k: v for k, v in r.items() if k not in ("logical_GBps",)})
    line["e2e"] = e2e
    line["gpu_launches"] = 2 * args.steps
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_line(cfg, args.cpu_budget, W.logical_bytes)
    line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def run_stream(args, dist, rank, world, local):
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    r = measure_stream(args, dev, local, world)
    line = base_line("c3", world, args, r["logical_GBps"], r["us_per_step"])
    line["steps"], line["warmup"] = r["decode_steps"], 0
    line.update({k: v for k, v in r.items() if k != "logical_GBps"})
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def run_sweep(args, dist, rank, local):
    torch.cuda.set_device(local)
    rows = codec_sweep(torch.device("cuda", local), [64 << k for k in range(7)])
    if rank == 0:
        print(json.dumps({"metric": "encode / standalone-decode GB/s sweep", "unit": "GB/s", "rows": rows,
                          "data": "synthetic", "flush": "L2 read-flushed before each call"}), flush=True)


def run_reference(args, dist, rank, world):
    """The CPU oracle as it stands, on the host cores, on the configuration the GPU arm
    measures: each step a bounded sample of that workload (sequences of one layer; for
    the 32-layer stack every layer has the same shape and distributions)."""
    if args.sweep or args.spread_sweep or args.format != "zf" or args.workload in ("c3", "serve"):
        sys.stderr.write("--impl reference times the CPU oracle on the attention workloads c2, c2-layer, c1 and c4 "
                         "only; it has no oracle counterpart for the requested mode\n")
        if dist:
            dist.destroy_process_group()
        sys.exit(2)
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    wl = args.workload
    cfg = layer_cfg("c2-layer" if wl == "c2" else wl)
    K, Wm = args.steps, args.warmup
    per_step_budget = max(0.5, min(4.0, 150.0 / max(1, K + Wm)))
    sample = OracleSample(cfg)  # the layer generated and encoded by the oracle once
    sample.size_for(per_step_budget, seqs_max=cfg.batch)
    vals, secs = [], []
    nseq = threads = 0
    for k in range(Wm + K):
        gbps, dt, nseq, passes, threads = sample.time(per_step_budget)
        if k >= Wm:
            vals.append(gbps)
            secs.append(dt)
    value = statistics.median(vals)
    lay = kvgen.gen_layout(cfg)
    layer_logical = kvgen.logical_kv_bytes(cfg, lay["seq_lens"])
    layers = kvgen.C2.layers if wl == "c2" else 1
    full_step_ms = layers * layer_logical / (value * 1e9) * 1e3
    logical_per_seq = (cfg.full_pages * 16 + (cfg.tail_min + cfg.tail_max) / 2) * cfg.hkv * 512
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": round(1e3 * statistics.median(secs), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(wl, world),
        "full_step_equivalent_ms": round(full_step_ms, 1),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "kind": "oracle", "cores": threads,
                         "sample": f"{nseq} sequence(s) x {cfg.hkv} KV heads of one layer per pass, repeated for "
                                   f"~{per_step_budget:.1f} s per step (~{nseq * logical_per_seq / 1e6:.0f} MB "
                                   "logical KV per pass); value = median over the steps"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="kvz", choices=["kvz", "reference"])
    ap.add_argument("--workload", default="c2", choices=["c2", "c2-layer", "c1", "c4", "c3", "serve"],
                    help="c2: the full 32-layer 8K step (default headline); c2-layer / c1 / c4: one layer as the "
                         "headline; c3: streaming decode with page-completion encodes; serve: toy admission loop")
    ap.add_argument("--no-extras", action="store_true",
                    help="c2: skip the extra keys (C1 layer, 8K layer, C4 layer and codec points, C3 streaming)")
    ap.add_argument("--serve-budget-gb", type=float, default=4.0, help="serve: KV budget of both caches (1e9 B)")
    ap.add_argument("--serve-requests", type=int, default=256, help="serve: requests in the queue")
    ap.add_argument("--budget-gb", type=float, default=60.0, help="KV budget for the c3 capacity count (1e9 B)")
    ap.add_argument("--sweep", action="store_true",
                    help="encode / standalone-decode throughput over 64 MB .. 4 GB of pages (exponent-spread KV)")
    ap.add_argument("--spread-sweep", action="store_true",
                    help="long-context layer (B=2, 131072 tokens) with the per-block exponent spread fixed at each "
                         "of 8..20: compressed fraction and attention time, compressed vs raw")
    ap.add_argument("--copies", type=int, default=3)
    ap.add_argument("--format", default="zf", choices=["zf", "ga", "f8e4", "f8e5"],
                    help="ga: group-adaptive additive tiles; f8e4 / f8e5: completed pages converted to FP8 "
                         "E4M3 / E5M2 and coded; instead of 12-bit block groups (c1, c2-layer, c4)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-steps", type=int, default=256, help="decode steps of the c3 streaming run")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    dist, rank, world, local = dist_setup()
    # the reference arm first: no GPU mode may run under its name
    if args.impl == "reference":
        return run_reference(args, dist, rank, world)
    if args.sweep:
        return run_sweep(args, dist, rank, local)
    if args.spread_sweep:
        return run_spread_sweep(args, dist, rank, local)
    if args.workload == "c3":
        return run_stream(args, dist, rank, world, local)
    if args.workload == "serve":
        return run_serve(args, dist, rank, world, local)
    if args.format != "zf":
        if args.workload == "c2":
            ap.error("the tile formats run on single layers: --workload c1, c2-layer or c4")
        return run_ga(args, layer_cfg(args.workload), dist, rank, world, local)
    if args.workload == "c2":
        return run_default(args, dist, rank, world, local)
    return run_layer(args, dist, rank, world, local)


if __name__ == "__main__":
    main()
