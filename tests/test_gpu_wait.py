"""The bounded barrier wait on the device (kvz_selftest_bounded_wait): a wait on a phase
nobody completes gives up after its limit with KVZ_STATUS_TIMEOUT and the kernel returns;
a wait on a completed phase returns at once; the context stays usable afterwards."""
import pytest
import torch

import kvgen
from helpers import Layer

pytestmark = pytest.mark.gpu


def test_wait_gives_up_after_its_limit_and_context_survives(oracle):
    import decode_attention_value_gb300 as kvz

    status = kvz.new_status()
    out = torch.zeros(3, dtype=torch.int64, device="cuda")
    limit = 50_000_000  # 50 ms
    kvz.selftest_bounded_wait(limit, status, out)
    torch.cuda.synchronize()
    first_ns, second_ns, flags = (int(x) for x in out.cpu())
    assert flags == 1, flags  # the completed phase succeeded, the dead one did not
    assert int(status.item()) == kvz.STATUS_TIMEOUT
    assert first_ns < 1_000_000
    assert limit <= second_ns < 20 * limit
    # the same context still runs the attention path correctly
    layer = Layer(kvgen.C0_TAIL, oracle)
    out_c = layer.run_compressed()
    out_r = layer.run_raw()
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    assert torch.equal(out_c, out_r)


def test_selftest_rejects_bad_limits():
    import decode_attention_value_gb300 as kvz

    status = kvz.new_status()
    out = torch.zeros(3, dtype=torch.int64, device="cuda")
    for bad in (0, 11_000_000_000):
        with pytest.raises(kvz.KvzError):
            kvz.selftest_bounded_wait(bad, status, out)
