"""SwiGLU folded into the down-projection's input transform (cuda-exl3 README,
"MoE throughput"), against the FP64 oracle: the transform alone, and a whole
gated MLP (gate_up GEMM -> fused SwiGLU transform -> down GEMM)."""
import numpy as np
import pytest
import torch

import exl3_trellis_quantized_gb300 as E
from exl3_trellis_quantized_gb300 import synthetic
from oracle import exl3_oracle as O
from oracle_check import assert_columns

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("m,k,s", [(37, 640, 2), (300, 1024, 1), (1, 256, 3)])
def test_swiglu_transform_parity(dtype, m, k, s):
    g = torch.Generator().manual_seed(6000 + m)
    gate_up = (torch.randn((m, 2 * k), generator=g) * 2.5).to(dtype)  # silu on both sides of zero
    suh = ((torch.rand((s, k), generator=g) * 0.4 + 0.8) * torch.sign(torch.randn((s, k), generator=g))).half()
    xh = E.input_transform_swiglu(gate_up.to(DEV), suh.to(DEV))
    torch.cuda.synchronize()
    got = _np(xh)
    ref = O.input_transform_swiglu(_np(gate_up), _np(suh))
    # fp32 path: silu (exp, add, divide) and the product with up and with suh,
    # each a few rounding steps of 2^-24, then 7 rounded butterfly stages over
    # the block: bound each output by 16 * 2^-24 of the block's absolute sum
    h = np.abs(O.swiglu(_np(gate_up)))
    terms = h[None] * np.abs(_np(suh))[:, None, :]
    blk_sum = np.repeat(terms.reshape(s, m, k // 128, 128).sum(-1), 128, axis=-1)
    e = 16 * 2.0 ** -24 * blk_sum * 2.0 ** -4
    lo = (ref - e).astype(np.float16).astype(np.float64)
    hi = (ref + e).astype(np.float16).astype(np.float64)
    bad = (got < lo) | (got > hi)
    assert not bad.any(), f"{bad.sum()} outside the rounding bracket"


def test_swiglu_empty_batch_and_rejections():
    suh = torch.ones((1, 256), dtype=torch.float16, device=DEV)
    out = E.input_transform_swiglu(torch.empty((0, 512), dtype=torch.bfloat16, device=DEV), suh)
    assert out.shape == (1, 0, 256)
    with pytest.raises(ValueError):
        E.input_transform_swiglu(torch.empty((4, 511), dtype=torch.bfloat16, device=DEV), suh)


def test_gated_mlp_chain():
    """gate_up (two shards of width I) -> fused SwiGLU transform -> down (split-k).
    The largest batch is checked against the oracle (run on the GPU's own gate_up
    output, column maxima over that batch); smaller batches must give the same
    rows byte for byte."""
    hidden, inter = 512, 768
    gu_layer = synthetic.make_layer(hidden, [inter, inter], 4, 1, seed=6100)
    dn_layer = synthetic.make_layer(inter, [hidden], 5, 2, seed=6101)
    x_all = synthetic.make_x(200, hidden, seed=6102)

    def mlp(m):
        gate_up = E.linear(x_all[:m].to(DEV), gu_layer.trellis.to(DEV), 4, 1, gu_layer.suh.to(DEV),
                           gu_layer.svh.to(DEV), gu_layer.shard_cols)
        xh = E.input_transform_swiglu(gate_up, dn_layer.suh.to(DEV))
        acc = torch.zeros(max(1, E.splitk_workspace_bytes(m, inter, hidden) // 4), dtype=torch.float32, device=DEV)
        y = E.gemm_splitk(xh, dn_layer.trellis.to(DEV), 5, 2, dn_layer.svh.to(DEV), dn_layer.shard_cols, acc)
        torch.cuda.synchronize()
        assert bool((acc == 0).all())
        return gate_up, y

    gate_up, y = mlp(200)
    h = O.swiglu(_np(gate_up))
    ref = O.linear(h, dn_layer.trellis.numpy(), 5, 2, _np(dn_layer.suh), _np(dn_layer.svh), dn_layer.shard_cols)
    got = _np(y)
    assert_columns(got, ref, "swiglu chain")
    for m in (1, 16):
        _, ym = mlp(m)
        assert torch.equal(ym.view(torch.int16), y[:m].view(torch.int16)), f"rows differ at m={m}"
    assert E.device_status() == 0
