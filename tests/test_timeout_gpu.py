"""The give-up path of the decode kernel's bounded waits, on the GPU.

Every wait inside the tensor-core decode kernel gives up after a time limit
(1 s by default): the kernel then records MLA_ERR_TIMEOUT in the device status
word, lets its in-flight copies land, waits for its tensor-core operations,
frees its tensor memory and returns.  The test lowers the limit through
mla_set_wait_limit_ns so that ordinary waits (a tile still loading, a message
still in flight) run out, checks that the status says so, then restores the
limit and checks that the next call on the same device returns the same bytes
as a call made before: nothing leaked (a CTA that kept its tensor memory would
make the next launch wait forever).  No fault, trap or endless wait is involved.
"""
import pytest
import torch

from head_latent_attention_23_b300 import mla, workloads as W
from head_latent_attention_23_b300.runner import DecodeStep

pytestmark = pytest.mark.gpu


def test_short_wait_limit_trips_and_the_next_call_recovers():
    w = W.cached_decode(8, [2048, 3000, 100, 4096, 777, 1500, 64, 2500], seed=41, permute=True)
    step = DecodeStep(w)
    if mla.decode_path(step.cfg) != 1:
        pytest.skip("the tensor-core decode kernel does not run on this device")
    step.run()
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK
    before = step.o_lat.clone()

    statuses = []
    mla.set_wait_limit_ns(1)
    try:
        for _ in range(3):
            step.decode()
            torch.cuda.synchronize()
            statuses.append(mla.get_status())
            if statuses[-1] == mla.MLA_ERR_TIMEOUT:
                break
    finally:
        mla.set_wait_limit_ns(0)
    assert mla.MLA_ERR_TIMEOUT in statuses, statuses

    step.decode()
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK
    assert torch.equal(step.o_lat, before)
