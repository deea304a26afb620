"""Mixture-of-experts path (cuda-exl3 README, "What is supported" and "MoE
notes"): the gathered per-expert input transform and the grouped GEMM over
block-aligned routed rows, against the FP64 oracle and against the dense path
run per expert."""
import numpy as np
import pytest
import torch

import exl3_trellis_quantized_gb300 as E
from exl3_trellis_quantized_gb300 import synthetic
from oracle import exl3_oracle as O

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL = 4e-3
SENTINEL = 0x7C01  # an fp16 NaN pattern nothing in the library writes


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


CASES = [
    # tokens, experts, topk, block, k, shard widths, bits, codebook
    (5, 8, 2, 32, 256, [256], 4, 1),
    (40, 6, 3, 32, 512, [256, 256], 3, 2),
    (70, 4, 2, 128, 256, [384], 6, 0),
    (300, 16, 4, 128, 384, [128, 128], 5, 1),
    (9, 5, 2, 32, 384, [256], 2, 0),  # odd k/128: 32-row blocks on two k atoms per stage
    (3, 6, 2, 32, 512, [384, 384], 4, 1),  # few blocks, 384-aligned shards: 96-column strips
    (4, 10, 2, 16, 256, [256], 4, 1),  # 16-row blocks (few tokens per expert)
    (7, 5, 3, 16, 384, [128, 128], 3, 2),  # 16-row blocks, odd k/128
]


def _setup(tokens, experts, topk, block, k, widths, bits, cb, seed):
    layer = synthetic.make_moe_layer(k, widths, bits, cb, experts, seed=seed)
    routing = synthetic.make_routing(tokens, experts, topk, block, seed=seed + 1)
    x = synthetic.make_x(tokens, k, seed=seed + 2)
    return layer, routing, x


@pytest.mark.parametrize("case", CASES, ids=[f"t{c[0]}e{c[1]}k{c[2]}b{c[3]}" for c in CASES])
def test_moe_input_transform(case):
    tokens, experts, topk, block, k, widths, bits, cb = case
    layer, r, x = _setup(*case, seed=7000 + tokens)
    s = len(widths)
    xh = torch.full((s, r.rows, k), SENTINEL, dtype=torch.int16, device=DEV).view(torch.float16)
    E.moe_input_transform(x.to(DEV), r.sorted_ids.to(DEV), topk, r.block_expert.to(DEV), block,
                          layer.suh.to(DEV), out=xh)
    torch.cuda.synchronize()
    ref = O.moe_input_transform(_np(x), r.sorted_ids.numpy(), r.block_expert.numpy(), block, topk,
                                _np(layer.suh))
    got = _np(xh)
    raw = xh.view(torch.int16).cpu().numpy()
    blocks = r.block_expert.numpy()
    live_rows = np.repeat(blocks >= 0, block)
    assert (raw[:, ~live_rows] == np.int16(SENTINEL)).all(), "rows of skipped blocks must not be written"
    # live rows: the plain transform's rounding bracket (exact products, 7 rounded adds)
    xs = np.zeros_like(ref)
    for row, pair in enumerate(r.sorted_ids.numpy()):
        if live_rows[row] and pair < tokens * topk:
            e = blocks[row // block]
            xs[:, row] = np.abs(_np(x)[pair // topk])[None] * np.abs(_np(layer.suh)[e])
    blk_sum = np.repeat(xs.reshape(s, r.rows, k // 128, 128).sum(-1), 128, axis=-1)
    e_b = 8 * 2.0 ** -24 * blk_sum * 2.0 ** -4
    lo = (ref - e_b).astype(np.float16).astype(np.float64)
    hi = (ref + e_b).astype(np.float16).astype(np.float64)
    sel = np.broadcast_to(live_rows[None, :, None], got.shape)
    bad = ((got < lo) | (got > hi)) & sel
    assert not bad.any(), f"{bad.sum()} live values outside the rounding bracket"


@pytest.mark.parametrize("case", CASES, ids=[f"t{c[0]}e{c[1]}k{c[2]}b{c[3]}" for c in CASES])
def test_moe_gemm(case):
    tokens, experts, topk, block, k, widths, bits, cb = case
    layer, r, x = _setup(*case, seed=7100 + tokens)
    n = sum(widths)
    tr, suh, svh = layer.trellis.to(DEV), layer.suh.to(DEV), layer.svh.to(DEV)
    ids, be = r.sorted_ids.to(DEV), r.block_expert.to(DEV)
    xh = E.moe_input_transform(x.to(DEV), ids, topk, be, block, suh)
    y = torch.full((r.rows, n), SENTINEL, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    E.moe_gemm(xh, tr, bits, cb, svh, layer.shard_cols, be, block, out=y)
    torch.cuda.synchronize()
    blocks = r.block_expert.numpy()
    raw = y.view(torch.int16).cpu().numpy()
    for b, e in enumerate(blocks):
        rows = slice(b * block, (b + 1) * block)
        if e < 0:
            assert (raw[rows] == np.int16(SENTINEL)).all(), f"block {b}: skipped block written"
            continue
        # the grouped rows are exactly the dense layer of this block's expert
        dense = E.gemm(xh[:, rows].contiguous(), tr[e].contiguous(), bits, cb, svh[e].contiguous(), layer.shard_cols)
        assert torch.equal(y[rows].view(torch.int16), dense.view(torch.int16)), f"block {b} differs from dense"
    ref = O.moe_linear(_np(x), r.sorted_ids.numpy(), blocks, block, topk, layer.trellis.numpy(), bits, cb,
                       _np(layer.suh), _np(layer.svh), layer.shard_cols)
    live = ~np.isnan(ref[:, 0])
    got = _np(y)[live]
    refl = ref[live]
    pad = r.sorted_ids.numpy()[live] >= tokens * topk
    assert (got[pad] == 0).all(), "padding rows must be zero"
    colmax = np.abs(refl).max(axis=0)
    assert np.all(np.abs(got - refl) <= TOL * colmax), f"worst {np.max(np.abs(got - refl) / colmax):.3e}"
    assert E.device_status() == 0


def test_moe_rejections():
    layer, r, x = _setup(5, 4, 2, 32, 256, [256], 4, 1, seed=7200)
    xh = E.moe_input_transform(x.to(DEV), r.sorted_ids.to(DEV), 2, r.block_expert.to(DEV), 32, layer.suh.to(DEV))
    with pytest.raises(E.Exl3Error):  # block size 64 is not supported
        E.moe_gemm(xh, layer.trellis.to(DEV), 4, 1, layer.svh.to(DEV), layer.shard_cols, r.block_expert.to(DEV), 64)
