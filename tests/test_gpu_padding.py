"""Padded dimensions (cuda-exl3 README, "Loading into a dim vLLM has padded").

Output side: a pad of whole 128-column blocks carries svh = 0, which makes those
columns exactly zero whatever the trellis behind them holds (the decoder is
total, so no pad code decodes to a NaN), and leaves the real columns untouched
because the Hadamard mixes only inside a 128-column block.

Input side: the producing layer's pad positions are exact zeros, so suh there
cannot reach the output, and zero input blocks add exact zeros to every sum.
The caller builds a padded-K layer from a checkpoint by copying the k16 tile
rows and suh entries that exist and zeroing the rest (the same page, "copy what
exists and zero the rest").
"""
import numpy as np
import pytest
import torch

import exl3_trellis_quantized_gb300 as E
from exl3_trellis_quantized_gb300 import synthetic
from oracle import exl3_oracle as O
from oracle_check import assert_columns, oracle_linear

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
    # the padded launch against the oracle of the padded layer (svh zero on the
    # pad); the column max is over the case's largest batch (300 rows, whose
    # prefix x is)
    ref_batch = oracle_linear(O, synthetic.make_x(300, k, seed=5101), padded, svh=svh.cpu())
    assert not ref_batch[:, n_real:].any()
    assert_columns(y.float().cpu().numpy(), ref_batch[:m], "padded output", ref_batch=ref_batch)
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


def pad_k_layer(trellis, suh, k_pad):
    """The caller's padded-K load: copy the k16 tile rows and suh entries that
    exist, zero the rest (the pad must be whole 128-row blocks)."""
    k_real = trellis.shape[0] * 16
    assert k_pad % 128 == 0 and k_real % 128 == 0 and k_pad >= k_real
    tr = torch.zeros((k_pad // 16,) + tuple(trellis.shape[1:]), dtype=trellis.dtype, device=trellis.device)
    tr[: k_real // 16] = trellis
    su = torch.zeros((suh.shape[0], k_pad), dtype=suh.dtype, device=suh.device)
    su[:, :k_real] = suh
    return tr, su


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("bits,cb,m", [(4, 1, 7), (6, 0, 130), (3, 2, 33)])
def test_padded_k_load_matches_oracle_of_unpadded_layer(bits, cb, m, split):
    """A checkpoint layer of K = 384 loaded into a dim padded to 640 (two whole
    pad blocks), fed activations whose pad positions are exact zeros (as the
    producing layer's padded output is): the output is the oracle's output of
    the unpadded layer, and the bytes of the unpadded launch."""
    k_real, k_pad, n = 384, 640, 256
    layer = synthetic.make_layer(k_real, [n], bits, cb, seed=5400 + bits)
    tr_pad, suh_pad = pad_k_layer(layer.trellis.to(DEV), layer.suh.to(DEV), k_pad)
    svh = layer.svh.to(DEV)
    x = synthetic.make_x(m, k_real, seed=5401).to(DEV)
    x_pad = torch.zeros((m, k_pad), dtype=x.dtype, device=DEV)
    x_pad[:, :k_real] = x

    def run(xx, tr, su):
        acc = None
        if split:
            acc = torch.zeros(max(1, E.splitk_workspace_bytes(m, xx.shape[1], n) // 4), dtype=torch.float32,
                              device=DEV)
        return E.linear(xx, tr, bits, cb, su, svh, layer.shard_cols, acc=acc)

    y_pad = run(x_pad, tr_pad, suh_pad)
    y_real = run(x, layer.trellis.to(DEV), layer.suh.to(DEV))
    torch.cuda.synchronize()
    ref_batch = oracle_linear(O, synthetic.make_x(130, k_real, seed=5401), layer)  # the case's largest batch
    assert_columns(y_pad.float().cpu().numpy(), ref_batch[:m], "padded-K load", ref_batch=ref_batch)
    if not split:  # the same k16 chain plus exact zeros
        assert torch.equal(y_pad.view(torch.int16), y_real.view(torch.int16))
    assert E.device_status() == 0
