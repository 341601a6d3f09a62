"""Parity at the benchmark's full sizes, in the launch configuration bench.py times:
the 131072-token long-context layer (every (sequence, KV head) unit split across ~29
CTAs, ~29 partials per merge) and the 8K-context layer, against the fp64 CPU oracle on
every output, plus sampled block tags and bit-exact standalone decodes of sampled pages."""
import numpy as np
import pytest
import torch

import kvgen
from helpers import check_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvz():
    from decode_attention_value_gb300 import _build

    _build.build()
    import decode_attention_value_gb300 as m

    return m


def _layer(kvz, cfg):
    """Device-generated layer, encoded on the GPU, as bench.Workload does (one copy)."""
    import bench

    return bench.Workload(cfg, 1, layer=0, dev=torch.device("cuda"))


def _oracle_attention(oracle, W, pick):
    cfg = W.cfg
    pool = kvgen.bits(W.pools[0].cpu())
    full = W.full[pick].cpu().numpy()
    per = (cfg.full_pages + 1) * cfg.hkv * 32
    o_meta = np.zeros((cfg.num_pages, cfg.hkv, 2), np.uint64)
    o_arena = np.zeros(len(pick) * per * 256, np.uint8)
    cur = np.array([[i * per, (i + 1) * per] for i in range(len(pick))], np.uint32)
    src = full.reshape(-1).astype(np.int32)
    seq = np.repeat(np.arange(len(pick), dtype=np.int32), cfg.full_pages)
    assert oracle.encode_pages(pool, src, src, seq, o_meta, o_arena, cur, cfg.hkv) == 0
    ref, st = oracle.decode_attention(kvgen.bits(W.q[pick].cpu()), full, W.seq_lens[pick].cpu().numpy(),
                                      W.tail[pick].cpu().numpy(), o_meta, o_arena, pool, cfg.hkv, nthreads=16)
    assert st == 0
    return ref, pool


def _check_blocks(kvz, oracle, W, pool, n_pages=48):
    """Sampled pages: GPU tags equal the oracle's, GPU decode returns the input bits."""
    cfg = W.cfg
    rng = np.random.default_rng(5)
    pages = rng.choice(W.src.cpu().numpy(), n_pages, replace=False).astype(np.int32)
    meta = W.metas[0].cpu().numpy().view(np.uint64)
    for p in pages[:12]:
        for h in range(cfg.hkv):
            for kv in range(2):
                tags = int(meta[p, h, kv]) >> 32
                for j in range(4):
                    _, t = oracle.encode_block(pool[p, h, kv], bool(kv), j)
                    assert ((tags >> (8 * j)) & 0xFF) == t
    out = torch.empty((n_pages, cfg.hkv, 2, 16, 128), dtype=torch.bfloat16, device="cuda")
    st = kvz.new_status()
    kvz.decode_blocks(W.metas[0], W.arenas[0], torch.from_numpy(pages).cuda(), out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), pool[pages])


def test_long_context_layer_all_outputs(kvz, oracle):
    cfg = kvgen.KVConfig(**{**kvgen.C4.__dict__, "layers": 1})
    W = _layer(kvz, cfg)
    W.step_c(0)
    W.step_r(0)
    torch.cuda.synchronize()
    assert int(W.status.item()) == 0
    assert torch.equal(W.out, W.out_raw)
    ref, pool = _oracle_attention(oracle, W, list(range(cfg.batch)))
    check_attention(W.out, ref, "long context")
    _check_blocks(kvz, oracle, W, pool)


def test_8k_layer_all_outputs(kvz, oracle):
    """One layer of the 8K stack (batch 16): every output against the oracle, and the
    decompress-first pipeline as bench.py times it equal to the fused kernel."""
    cfg = kvgen.KVConfig(**{**kvgen.C2.__dict__, "layers": 1})
    W = _layer(kvz, cfg)
    W.step_c(0)
    W.step_r(0)
    W.setup_decompress_first()
    W.step_df(0)
    torch.cuda.synchronize()
    assert int(W.status.item()) == 0
    assert torch.equal(W.out, W.out_raw)
    assert torch.equal(W.out_df, W.out)
    ref, pool = _oracle_attention(oracle, W, list(range(cfg.batch)))
    check_attention(W.out, ref, "8K layer")
    _check_blocks(kvz, oracle, W, pool)


def test_c1_layer_decompress_first_all_outputs(kvz, oracle):
    """The C1 layer's decompress-first pipeline (standalone decode into a BF16 scratch
    pool, then the raw kernel), as bench.py times it: every output against the oracle."""
    W = _layer(kvz, kvgen.C1)
    W.setup_decompress_first()
    W.step_df(0)
    W.step_c(0)
    torch.cuda.synchronize()
    assert int(W.status.item()) == 0
    assert torch.equal(W.out_df, W.out)
    ref, _ = _oracle_attention(oracle, W, list(range(W.cfg.batch)))
    check_attention(W.out_df, ref, "C1 decompress-first")


@pytest.mark.parametrize("kind", ["ga", "f8e4", "f8e5"])
def test_c1_tile_formats_sampled(kvz, oracle, kind):
    """The tile formats on the Llama-3.1-8B-shaped layer in the launch configuration
    bench.py --format times: bases calibrated on the GPU equal the oracle's own (same
    sample of pages), and sampled sequences' outputs match the fp64 oracle run over the
    oracle's own tiles of those sequences."""
    import bench

    W = _layer(kvz, kvgen.C1)
    GA = bench.GaCopies(W, kind)
    GA.step(0)
    torch.cuda.synchronize()
    assert int(W.status.item()) == 0
    cfg, hkv = W.cfg, W.cfg.hkv
    pool = kvgen.bits(W.pools[0].cpu())
    sample = GA.sample.cpu().numpy().astype(np.int32)
    fmt = {"f8e4": 1, "f8e5": 2}.get(kind)
    o_bases = (oracle.ga_calibrate_pool(pool, sample, hkv) if kind == "ga"
               else oracle.f8_calibrate_pool(fmt, pool, sample, hkv))
    assert np.array_equal(GA.bases.cpu().numpy(), o_bases), "bases"
    pick = [0, 13, 31]
    full = W.full[pick].cpu().numpy()
    gran = (64 if kind == "ga" else 32) * hkv * 2  # worst-case 64-byte granules per page
    per = cfg.full_pages * gran
    o_meta = np.zeros((cfg.num_pages, hkv, 2), np.uint32)
    o_arena = np.zeros(len(pick) * per * 64, np.uint8)
    cur = np.array([[i * per, (i + 1) * per] for i in range(len(pick))], np.uint32)
    src = full.reshape(-1).astype(np.int32)
    seq = np.repeat(np.arange(len(pick), dtype=np.int32), cfg.full_pages)
    q = kvgen.bits(W.q[pick].cpu())
    lens, tail = W.seq_lens[pick].cpu().numpy(), W.tail[pick].cpu().numpy()
    if kind == "ga":
        assert oracle.ga_encode_pages(pool, o_bases, src, src, seq, o_meta, o_arena, cur, hkv) == 0
        ref, st = oracle.ga_decode_attention(q, full, lens, tail, o_meta, o_arena, o_bases, pool, hkv, nthreads=16)
    else:
        assert oracle.f8_encode_pages(fmt, pool, o_bases, src, src, seq, o_meta, o_arena, cur, hkv) == 0
        ref, st = oracle.f8_decode_attention(fmt, q, full, lens, tail, o_meta, o_arena, o_bases, pool, hkv,
                                             nthreads=16)
    assert st == 0
    check_attention(GA.out[pick], ref, f"C1 {kind}")
