"""Padded dimensions (cuda-exl3 README, "Loading into a dim vLLM has padded").

Output side: a pad of whole 128-column blocks carries svh = 0, which makes those
columns exactly zero whatever the trellis behind them holds (the decoder is
total, so no pad code decodes to a NaN), and leaves the real columns untouched
because the Hadamard mixes only inside a 128-column block.

Input side: the producing layer's pad positions are exact zeros, so suh there
cannot reach the output, and zero input blocks add exact zeros to every sum.
"""
import numpy as np
import pytest
import torch

import exl3_trellis_quantized_gb300 as E
from exl3_trellis_quantized_gb300 import synthetic

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _dev(layer):
    return layer.trellis.to(DEV), layer.suh.to(DEV), layer.svh.to(DEV)


@pytest.mark.parametrize("cb", [0, 1, 2])
@pytest.mark.parametrize("m", [3, 300])
def test_output_pad_blocks_are_exact_zeros(cb, m):
    k, n_real, n_pad, bits = 512, 384, 640, 4
    padded = synthetic.make_layer(k, [n_pad], bits, cb, seed=5100 + cb)
    tr, suh, svh = _dev(padded)
    svh = svh.clone()
    svh[n_real:] = 0  # the pad: two whole 128-column blocks
    x = synthetic.make_x(m, k, seed=5101).to(DEV)
    xh = E.input_transform(x, suh)
    y = E.gemm(xh, tr, bits, cb, svh, [0, n_pad])
    torch.cuda.synchronize()
    assert bool((y[:, n_real:].float() == 0).all()), "pad columns must be exactly zero"
    # the real columns equal a launch over the real columns alone
    tr_real = tr[:, : n_real // 16].contiguous()
    y_real = E.gemm(xh, tr_real, bits, cb, svh[:n_real].contiguous(), [0, n_real])
    assert torch.equal(y[:, :n_real].contiguous().view(torch.int16), y_real.view(torch.int16))
    assert E.device_status() == 0


def test_input_pad_zeros_hide_suh():
    """x is zero on the pad positions: any suh there gives the same xh values."""
    k, m = 512, 37
    x = synthetic.make_x(m, k, seed=5200).to(DEV)
    x[:, 300:] = 0  # pad inside the third block and the whole fourth block
    g = torch.Generator().manual_seed(5201)
    suh_a = (torch.rand(1, k, generator=g) + 0.5).half().to(DEV)
    suh_b = suh_a.clone()
    suh_b[:, 300:] = -7.0  # different scales on the pad only
    xa = E.input_transform(x, suh_a)
    xb = E.input_transform(x, suh_b)
    # equal values; only the sign of an exact zero may follow the pad's suh
    # (0 * -7 is -0), so compare numbers, not bit patterns
    assert torch.equal(xa.float(), xb.float())


@pytest.mark.parametrize("m", [5, 200])
def test_input_pad_blocks_add_exact_zeros(m):
    """A layer padded from k=256 to k=512 with zero inputs on the pad gives the
    bytes of the unpadded layer (the extra k16 steps add exact zeros)."""
    k_real, k_pad, n, bits, cb = 256, 512, 256, 5, 1
    layer = synthetic.make_layer(k_pad, [n], bits, cb, seed=5300)
    tr, suh, svh = _dev(layer)
    x = synthetic.make_x(m, k_pad, seed=5301).to(DEV)
    x[:, k_real:] = 0
    y_pad = E.gemm(E.input_transform(x, suh), tr, bits, cb, svh, [0, n])
    x_real = x[:, :k_real].contiguous()
    tr_real = tr[: k_real // 16].contiguous()
    y_real = E.gemm(E.input_transform(x_real, suh[:, :k_real].contiguous()), tr_real, bits, cb, svh, [0, n])
    assert torch.equal(y_pad.view(torch.int16), y_real.view(torch.int16))
    assert np.isfinite(y_pad.float().cpu().numpy()).all()
