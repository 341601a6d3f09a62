"""The fill-then-finalize lifecycle (GAAC "Block-Wise Compression Scheduling"; the
ZipFusion memory manager) through decode_attention_value_gb300.cache: sequences are
admitted with a prefill-side bulk encode, grow a token per step with their pages encoded
as they fill, and are released so their arena chunks serve later sequences.  The
compressed cache and a raw cache are driven in lockstep with the same KV; every step their
attention outputs must be bit-identical, and at sampled steps both match the fp64 oracle
over a host copy of each sequence's KV."""
import dataclasses

import numpy as np
import pytest
import torch

import kvgen
from helpers import check_attention

pytestmark = pytest.mark.gpu


def test_lockstep_lifecycle_with_chunk_recycling(oracle):
    import decode_attention_value_gb300 as kvz
    from decode_attention_value_gb300.cache import CompressedKVCache, RawKVCache

    L, hkv, hq, max_seqs, max_pages = 2, 2, 8, 6, 12
    cfg = dataclasses.replace(kvgen.C1, hkv=hkv, hq=hq, batch=max_seqs, seed=91)
    rng = np.random.default_rng(91)
    # 64 KB chunks (256 granules): one sequence fills several and frees them on release
    comp = CompressedKVCache(L, hkv, max_seqs, max_pages, arena_bytes=40 * 256 * 256, chunk_granules=256)
    raw = RawKVCache(L, hkv, max_seqs, max_pages, num_slots=max_seqs * (max_pages + 1))
    sig = [kvgen.channel_sigmas(cfg, layer, "cuda") for layer in range(L)]
    qs = [torch.randn((max_seqs, hq, 128), device="cuda").to(torch.bfloat16) for _ in range(L)]
    mirror = {}  # slot -> [L][tokens][hkv][2][128] host BF16 bits
    requests = [(int(rng.integers(17, 120)), int(rng.integers(5, 60))) for _ in range(14)]
    queue, running, free = list(range(len(requests))), {}, list(range(max_seqs))
    step, checked = 0, 0
    out_c = torch.empty((max_seqs, hq, 128), dtype=torch.float32, device="cuda")
    out_r = torch.empty_like(out_c)
    ws = comp.workspace(max_seqs, hq)
    while queue or running:
        while queue and free and len(running) < 4:
            rid = queue.pop(0)
            slot = free.pop()
            n_tok, gen = requests[rid]
            n_pages = (n_tok + 15) // 16
            prompt = torch.stack([kvgen.gen_pages(cfg, n_pages, layer=layer, device="cuda", seed_offset=977 * rid)
                                  for layer in range(L)])
            # tokens past the prompt length in the last page are not part of the sequence
            comp.admit(slot, prompt, n_tok)
            raw.admit(slot, prompt, n_tok)
            m = prompt.permute(0, 1, 4, 2, 3, 5).reshape(L, n_pages * 16, hkv, 2, 128)[:, :n_tok]
            mirror[slot] = [kvgen.bits(m[layer].cpu()) for layer in range(L)]
            running[slot] = [rid, gen]
        slots = sorted(running)
        x = torch.randn((L, len(slots), hkv, 2, 128), device="cuda")
        for layer in range(L):
            ks, vs = sig[layer]
            x[layer, :, :, 0] *= ks
            x[layer, :, :, 1] *= vs
        kv = x.to(torch.bfloat16)
        comp.append(slots, kv)
        raw.append(slots, kv)
        kv_bits = kvgen.bits(kv.cpu())
        for i, s in enumerate(slots):
            for layer in range(L):
                mirror[s][layer] = np.concatenate([mirror[s][layer], kv_bits[layer, i][None]], 0)
        a_c, a_r = comp.batch_args(slots), raw.batch_args(slots)
        n = len(slots)
        for layer in range(L):
            comp.attention(layer, qs[layer][:n].contiguous(), a_c, out_c[:n], workspace=ws)
            raw.attention(layer, qs[layer][:n].contiguous(), a_r, out_r[:n], workspace=ws)
            torch.cuda.synchronize()
            assert int(comp.status.item()) == 0 and int(raw.status.item()) == 0
            assert torch.equal(out_c[:n], out_r[:n]), f"step {step} layer {layer}"
            if step % 9 == 0:
                # oracle over the mirrored KV: each sequence's tokens as plain pages
                pool, table, lens = [], [], []
                for s in slots:
                    t = mirror[s][layer]
                    npg = (t.shape[0] + 15) // 16
                    pad = np.zeros((npg * 16 - t.shape[0],) + t.shape[1:], np.uint16)
                    pg = np.concatenate([t, pad], 0).reshape(npg, 16, hkv, 2, 128).transpose(0, 2, 3, 1, 4)
                    table.append(list(range(len(pool), len(pool) + npg)))
                    pool.extend(pg)
                    lens.append(t.shape[0])
                width = max(len(r) for r in table)
                tab = np.array([r + [-1] * (width - len(r)) for r in table], np.int32)
                ref, st = oracle.attention_raw(kvgen.bits(qs[layer][:n].cpu()), tab, np.array(lens, np.int32),
                                               np.ascontiguousarray(np.stack(pool)), hkv)
                assert st == 0
                check_attention(out_c[:n], ref, f"step {step} layer {layer}")
                checked += 1
        for s in slots:
            running[s][1] -= 1
            if running[s][1] == 0:
                comp.release(s)
                raw.release(s)
                del running[s], mirror[s]
                free.append(s)
        step += 1
    assert checked >= 6
    st = comp.stats()
    assert st["chunks_held"] == 0 and st["chunks_free"] == 40  # everything came back
    assert comp.chunk_grants > 40  # more chunk hand-outs than the arena has: released chunks were reused


def test_compressed_cache_reports_out_of_space_without_changes():
    import decode_attention_value_gb300 as kvz
    from decode_attention_value_gb300.cache import CompressedKVCache, OutOfSpace

    L, hkv = 2, 2
    cfg = dataclasses.replace(kvgen.C1, hkv=hkv, hq=8, batch=2, seed=92)
    # three 64 KB chunks; the worst case of a (page, layer) is 64 granules of 256 B
    comp = CompressedKVCache(L, hkv, 2, 8, arena_bytes=3 * 256 * 256, chunk_granules=256)
    prompt = torch.stack([kvgen.gen_pages(cfg, 3, layer=layer, device="cuda") for layer in range(L)])
    comp.admit(0, prompt, 47)  # two full pages per layer (~215 of 256 granules), 15-token tail
    comp.admit(1, prompt, 47)  # the second chunk
    lens_before = comp.lens.copy()
    tails_before = comp.tails.clone()
    kv = torch.zeros((L, 2, hkv, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(OutOfSpace):
        comp.append([0, 1], kv)  # both tails fill: each needs a fresh chunk, one is left
    assert np.array_equal(comp.lens, lens_before)
    assert torch.equal(comp.tails, tails_before)
    torch.cuda.synchronize()
    assert int(comp.status.item()) == 0
