"""kvz_decode_attention_noalloc: the attention entry point for callers that cannot
allocate device memory (their framework owns every device allocation, or their
policy forbids allocation while work is recorded).  It keeps its split-KV scratch in
a fixed array inside libkvz instead of a caller workspace.

Called here through the C ABI with ctypes, twice in a row (the second call finds the
first call's leftovers in the shared array).  Both calls use the same work split as
kvz_decode_attention, so their outputs must equal its output bit for bit; they are also
checked against the fp64 CPU oracle within the attention tolerance of the other GPU
tests.  The file name makes pytest collect it last."""
import ctypes

import numpy as np
import pytest
import torch

import kvgen
from helpers import Layer, check_attention

pytestmark = pytest.mark.gpu


def _noalloc_fn(kvz):
    lib = ctypes.CDLL(kvz._build.LIB)
    fn = lib.kvz_decode_attention_noalloc
    P, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
    fn.restype = ctypes.c_int
    fn.argtypes = [kvz.Dims, i32, i32, P, P, i32, P, P, P, i64, P, u64, P, i64, P, P, P]
    return fn


def _call(kvz, fn, layer, out, status, batch=None):
    cfg = layer.cfg
    hkv = cfg.hkv
    # keep the device copies referenced until the call has been enqueued: a dropped
    # temporary's block can be handed to the next allocation
    full, lens, tail = layer.full.cuda(), layer.seq_lens.cuda(), layer.tail.cuda()
    return fn(kvz.Dims(hkv, 128, 16), cfg.batch if batch is None else batch, cfg.hq, layer.g_q.data_ptr(),
              full.data_ptr(), full.shape[1], lens.data_ptr(), tail.data_ptr(),
              layer.meta.data_ptr(), layer.meta.shape[0], layer.arena.data_ptr(), layer.arena.numel(),
              layer.g_pool.data_ptr(), layer.g_pool.shape[0], out.data_ptr(), status.data_ptr(),
              torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point(oracle):
    import decode_attention_value_gb300 as kvz

    fn = _noalloc_fn(kvz)
    cfg = kvgen.KVConfig("noalloc-ragged", 1, 12, 32, 8, 40, tail_min=1, tail_max=15, k_log2_sigma=(-4, 3),
                         v_log2_sigma=(-3, 1), k_outlier_channels=4, k_outlier_scale=32.0, seed=77)
    rng = np.random.default_rng(77)
    lens = rng.integers(0, 40 * 16 + 16, cfg.batch).astype(np.int32)
    lens[3] = 0
    lens[5] = 16 * 7  # a whole number of pages: no tail
    layer = Layer(cfg, oracle, seq_lens=lens)
    ref = layer.run_compressed()
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    o_ref, o_st = layer.oracle_attention(oracle)
    assert o_st == 0
    check_attention(ref, o_ref, "workspace entry point")
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        status = kvz.new_status()
        rc = _call(kvz, fn, layer, out, status)
        assert rc == 0, kvz.lib().kvz_strerror(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: status {int(status.item())}"
        assert torch.equal(out, ref), f"call {call}: differs from kvz_decode_attention"
        check_attention(out, o_ref, f"no-alloc call {call}")


def test_noalloc_rejects_problems_beyond_its_array():
    import decode_attention_value_gb300 as kvz

    fn = _noalloc_fn(kvz)
    layer = Layer(kvgen.C0_TAIL, None)
    out = torch.empty((256, 32, 128), dtype=torch.float32, device="cuda")
    status = kvz.new_status()
    full, lens, tail = layer.full.cuda(), layer.seq_lens.cuda(), layer.tail.cuda()
    # 256 sequences x 8 KV heads needs more split scratch than the fixed array holds;
    # the call must refuse on the host, before anything is launched
    rc = fn(kvz.Dims(8, 128, 16), 256, 32, layer.g_q.data_ptr(), full.data_ptr(), 1,
            lens.data_ptr(), tail.data_ptr(), layer.meta.data_ptr(), 1,
            layer.arena.data_ptr(), layer.arena.numel(), layer.g_pool.data_ptr(), 1, out.data_ptr(),
            status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == -8, kvz.lib().kvz_strerror(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
