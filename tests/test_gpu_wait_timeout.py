"""The failure path of the kernels' bounded waits, taken on purpose and
without a fault: a kernel waits on an mbarrier that nothing arrives on, gives
up after 2 s, records the wait-timeout flag and returns; the flag reads back
once through exl3_device_status, and the context stays usable."""
import pytest
import torch

import exl3_trellis_quantized_gb300 as E
from exl3_trellis_quantized_gb300 import binding as B
from exl3_trellis_quantized_gb300 import synthetic

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
WAIT_TIMEOUT = 1  # EXL3_DEVERR_WAIT_TIMEOUT


def _layer_call():
    layer = synthetic.make_layer(512, [256], 4, 1, seed=4900)
    x = synthetic.make_x(16, 512, seed=4901).to(DEV)
    xh = E.input_transform(x, layer.suh.to(DEV))
    return E.gemm(xh, layer.trellis.to(DEV), 4, 1, layer.svh.to(DEV), layer.shard_cols)


def test_bounded_wait_gives_up_and_reports():
    before = _layer_call()
    assert B.device_status() == 0
    assert B.test_wait_timeout() == 0, "the wait returned although nothing arrived"
    assert B.device_status() == WAIT_TIMEOUT
    assert B.device_status() == 0, "reading the flags clears them"
    after = _layer_call()
    torch.cuda.synchronize()
    assert torch.equal(before.view(torch.int16), after.view(torch.int16)), "the context is no longer usable"
    assert B.device_status() == 0
