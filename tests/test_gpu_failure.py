"""Failure detection on the GPU without a fault: a device wait that cannot
complete gives up after its limit, records CSA_ERR_TIMEOUT in the status word,
stops the other waits of its CTA through the abort flag, and leaves the
context usable for the next call."""
import pytest
import torch

from long_context_compressed_18_b300 import inputs, lib
from helpers import DEV

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_stays_usable():
    torch.cuda.synchronize()
    lib.csa_device_status()                          # start from a clear word
    aborted = torch.zeros(4, dtype=torch.int32, device=DEV)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    lib.csa_wait_selftest(2000, aborted)             # a 2 ms limit on a wait nothing completes
    e1.record()
    with pytest.raises(lib.CsaError) as e:
        lib.csa_device_status()
    assert e.value.status == 6                       # CSA_ERR_TIMEOUT
    assert int(aborted[0].item()) == 1               # the second warp stopped on the abort flag
    ms = e0.elapsed_time(e1)
    assert 1.5 <= ms < 1000.0, ms                    # gave up after its own limit, not the 2 s default
    lib.csa_device_status()                          # read-and-clear: the word is clear again

    # the same context runs a normal call correctly afterwards
    sc = inputs.random_scores(3, 5000, seed=5).to(DEV)
    out = torch.empty(3, 64, dtype=torch.int32, device=DEV)
    lib.csa_topk_select(3, 1, 4 * 5000 - 1, 4, 5000, 64, sc, out)
    torch.cuda.synchronize()
    lib.csa_device_status()
    want = torch.topk(sc.cpu(), 64, dim=1).indices.sort(dim=1).values.to(torch.int32)
    assert torch.equal(out.cpu(), want)


def test_wait_selftest_rejects_bad_limits_on_the_host():
    aborted = torch.zeros(4, dtype=torch.int32, device=DEV)
    for bad in (0, 2000001):
        with pytest.raises(lib.CsaError) as e:
            lib.csa_wait_selftest(bad, aborted)
        assert e.value.status == 1
