"""Overlapped attention launches (KVZ_ATTN_OVERLAP_PREVIOUS): the attention kernel starts
while the kernel before it is still running, reads lengths, tables, metadata and the
compressed (or non-last raw) pages early, and reads q and each sequence's last page only
after that kernel has finished.  Checked: outputs bit-identical to the plain calls, and
a late writer (a kernel that lets the dependent launch begin, waits, then writes q or
the last page) never leaves its old values in the result, eagerly and in a CUDA graph."""
import pytest
import torch

import kvgen
from helpers import Layer, check_attention

pytestmark = pytest.mark.gpu

OVER = 1  # KVZ_ATTN_OVERLAP_PREVIOUS
DELAY_NS = 50_000  # the late writer's wait: far longer than the attention kernel's start-up


@pytest.fixture(scope="module")
def kvz():
    from decode_attention_value_gb300 import _build

    _build.build()
    import decode_attention_value_gb300 as m

    return m


class Args:
    """Device copies of a layer's call arguments, made before any timed or overlapped
    sequence: a host-to-device copy between the late writer and the attention launch
    would sit between them on the stream and turn the programmatic dependency into a
    plain one."""

    def __init__(self, layer):
        self.full, self.lens, self.tail = layer.full.cuda(), layer.seq_lens.cuda(), layer.tail.cuda()
        self.raw_table = layer.raw_table().cuda()
        self.ws_c, self.ws_r = layer.workspace(False), layer.workspace(True)
        torch.cuda.synchronize()


def _attend(kvz, layer, a, q, flags, out_c=None, out_r=None, status=None):
    if out_c is not None:
        kvz.decode_attention(q, a.full, a.lens, a.tail, layer.meta, layer.arena, layer.g_pool, out_c, status,
                             workspace=a.ws_c, flags=flags)
    if out_r is not None:
        kvz.decode_attention_raw(q, a.raw_table, a.lens, layer.g_pool, out_r, status, workspace=a.ws_r, flags=flags)


CASES = [
    kvgen.C0_TAIL,
    kvgen.KVConfig("ragged-b6", 1, 6, 16, 4, 9, tail_min=1, tail_max=15, k_log2_sigma=(-4, 3), v_log2_sigma=(-3, 1),
                   k_outlier_channels=4, k_outlier_scale=32.0, block_outlier_frac=0.05, seed=31),
    kvgen.KVConfig("gqa8", 1, 5, 16, 2, 11, tail_min=1, tail_max=15, seed=36),
    kvgen.KVConfig("long", 1, 2, 8, 2, 300, tail_min=5, tail_max=11, seed=42),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_overlap_matches_plain_calls(kvz, oracle, cfg):
    layer = Layer(cfg, oracle)
    a = Args(layer)
    shape = (cfg.batch, cfg.hq, 128)
    outs = {k: torch.empty(shape, dtype=torch.float32, device="cuda") for k in ("c0", "r0", "c1", "r1")}
    st = kvz.new_status()
    _attend(kvz, layer, a, layer.g_q, 0, outs["c0"], outs["r0"], st)
    # overlapped calls back to back: each also overlaps the previous call's merge
    _attend(kvz, layer, a, layer.g_q, OVER, outs["c1"], outs["r1"], st)
    _attend(kvz, layer, a, layer.g_q, OVER, outs["c1"], outs["r1"], st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for k in ("c1", "r1"):
        assert torch.equal(outs[k], outs["c0"]), k
    assert torch.equal(outs["r0"], outs["c0"])
    ref, ost = layer.oracle_attention(oracle)
    assert ost == 0
    check_attention(outs["c1"], ref, cfg.name + " overlapped")


def _late_q_step(kvz, layer, a, q_buf, q_true, out_c, out_r, st):
    kvz.selftest_late_writer(q_true, q_buf, DELAY_NS)
    _attend(kvz, layer, a, q_buf, OVER, out_c=out_c, status=st)
    kvz.selftest_late_writer(q_true, q_buf, DELAY_NS)
    _attend(kvz, layer, a, q_buf, OVER, out_r=out_r, status=st)


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
def test_overlap_reads_q_after_the_previous_kernel(kvz, oracle, graph):
    cfg = CASES[1]
    layer = Layer(cfg, oracle)
    a = Args(layer)
    ref = layer.run_compressed()
    torch.cuda.synchronize()
    q_true = layer.g_q.clone()
    q_buf = torch.zeros_like(q_true)  # what an early read would see
    out_c, out_r = torch.full_like(ref, float("nan")), torch.full_like(ref, float("nan"))
    st = kvz.new_status()
    if graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            _late_q_step(kvz, layer, a, q_buf, q_true, out_c, out_r, st)  # warm-up: configures the kernels
            torch.cuda.synchronize()
            q_buf.zero_()
            with torch.cuda.graph(g, stream=s):
                _late_q_step(kvz, layer, a, q_buf, q_true, out_c, out_r, st)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        for _ in range(2):
            q_buf.zero_()
            out_c.fill_(float("nan"))
            out_r.fill_(float("nan"))
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(out_c, ref) and torch.equal(out_r, ref)
    else:
        _late_q_step(kvz, layer, a, q_buf, q_true, out_c, out_r, st)
        torch.cuda.synchronize()
        assert torch.equal(out_c, ref) and torch.equal(out_r, ref)
    assert int(st.item()) == 0


def test_overlap_reads_the_last_page_after_the_previous_kernel(kvz, oracle):
    """One sequence whose last page (16 KB: both KV heads, K and V) is rewritten by the
    late writer; the overlapped calls must attend over the new values."""
    cfg = kvgen.C0_TAIL
    layer = Layer(cfg, oracle)
    tail = int(layer.tail[0])
    ref = layer.run_compressed()
    torch.cuda.synchronize()
    page_true = layer.g_pool[tail].clone()
    layer.g_pool[tail].zero_()  # what an early read would see (a zero last page changes the output)
    stale = layer.run_compressed()
    torch.cuda.synchronize()
    assert not torch.equal(stale, ref)
    a = Args(layer)
    out_c, out_r = torch.full_like(ref, float("nan")), torch.full_like(ref, float("nan"))
    st = kvz.new_status()
    for call in ("c", "r"):
        layer.g_pool[tail].zero_()
        kvz.selftest_late_writer(page_true, layer.g_pool[tail], DELAY_NS)
        if call == "c":
            _attend(kvz, layer, a, layer.g_q, OVER, out_c=out_c, status=st)
        else:
            _attend(kvz, layer, a, layer.g_q, OVER, out_r=out_r, status=st)
        torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out_c, ref) and torch.equal(out_r, ref)


def test_overlap_flag_checks(kvz):
    lib = kvz.lib()
    fake = 1 << 20
    d = kvz.Dims(8, 128, 16)
    # unknown flag bits are refused on the host
    assert lib.kvz_decode_attention_ex(d, 2, 32, fake, fake, 4, fake, fake, fake, 1, fake, 1 << 20, fake, 1, fake,
                                       fake, 1 << 20, fake, 2, None) == -1
    assert lib.kvz_decode_attention_raw_ex(d, 2, 32, fake, fake, 4, fake, fake, 1, fake, fake, 1 << 20, fake, 4,
                                           None) == -1
    assert lib.kvz_selftest_late_writer(fake, fake + 8, 16, 0, None) == -3
    assert lib.kvz_selftest_late_writer(fake, fake, 16, 2_000_000_000, None) == -1
