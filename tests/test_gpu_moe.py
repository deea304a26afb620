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
from oracle_check import assert_columns

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
    (60, 4, 2, 128, 512, [256], 8, 1),  # 128-row blocks at 8 bits: two k atoms a stage
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
    assert_columns(got, refl, "moe linear")
    assert E.device_status() == 0


def test_moe_rejections():
    layer, r, x = _setup(5, 4, 2, 32, 256, [256], 4, 1, seed=7200)
    xh = E.moe_input_transform(x.to(DEV), r.sorted_ids.to(DEV), 2, r.block_expert.to(DEV), 32, layer.suh.to(DEV))
    with pytest.raises(E.Exl3Error):  # block size 64 is not supported
        E.moe_gemm(xh, layer.trellis.to(DEV), 4, 1, layer.svh.to(DEV), layer.shard_cols, r.block_expert.to(DEV), 64)


# ---------------------------------------------------------------------------
# The weighted combine of each token's top-k rows (exl3_moe_combine)
# ---------------------------------------------------------------------------

COMBINE_CASES = [CASES[0], CASES[1], CASES[3], CASES[6]]
BF16_NAN = 0x7FC1  # a bf16 NaN pattern: rows of skipped blocks keep it, so reading one would show


def _routed_rows(layer, r, x, tokens, topk, block, block_expert):
    """The grouped GEMM's output on the GPU, skipped blocks' rows left as NaN."""
    tr, suh, svh = layer.trellis.to(DEV), layer.suh.to(DEV), layer.svh.to(DEV)
    ids, be = r.sorted_ids.to(DEV), block_expert.to(DEV)
    xh = E.moe_input_transform(x.to(DEV), ids, topk, be, block, suh)
    y = torch.full((r.rows, layer.n), BF16_NAN, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    E.moe_gemm(xh, tr, layer.bits, layer.codebook, svh, layer.shard_cols, be, block, out=y)
    return y, ids, be


@pytest.mark.parametrize("case", COMBINE_CASES, ids=[f"t{c[0]}e{c[1]}k{c[2]}b{c[3]}" for c in COMBINE_CASES])
@pytest.mark.parametrize("drop", [False, True], ids=["all", "dropped_block"])
def test_moe_combine_against_oracle(case, drop):
    """The whole routed layer plus combine against the oracle.  Each routed row
    meets the per-column bar on its own; the combine's weights sum to 1, so the
    error of a token is at most the weighted sum of its rows' bars plus the
    final bf16 rounding (2^-8 relative, with margin for fp32 sums)."""
    tokens, experts, topk, block, k, widths, bits, cb = case
    layer, r, x = _setup(*case, seed=7300 + tokens)
    be_host = r.block_expert.clone()
    if drop:  # a live block marked as no expert: its pairs' terms disappear
        be_host[int(torch.nonzero(be_host >= 0)[0])] = -1
    y, ids, be = _routed_rows(layer, r, x, tokens, topk, block, be_host)
    w = synthetic.make_topk_weights(tokens, topk, seed=7301 + tokens)
    out = E.moe_combine(y, ids, be, block, experts, w.to(DEV), topk)
    torch.cuda.synchronize()
    rows = O.moe_linear(_np(x), r.sorted_ids.numpy(), be_host.numpy(), block, topk, layer.trellis.numpy(), bits, cb,
                        _np(layer.suh), _np(layer.svh), layer.shard_cols)
    ref = O.moe_combine(rows, r.sorted_ids.numpy(), be_host.numpy(), block, topk, w.double().numpy(), tokens,
                        experts)
    got = _np(out)
    assert np.isfinite(got).all(), "a padding row or a skipped block's row was read"
    colmax = np.nanmax(np.abs(rows), axis=0)  # each routed row's per-column bar is TOL * colmax
    wsum = np.zeros(tokens)
    ids_np = r.sorted_ids.numpy()
    live = np.repeat(be_host.numpy() >= 0, block)
    for row, pair in enumerate(ids_np):
        if live[row] and pair < tokens * topk:
            t, j = divmod(int(pair), topk)
            wsum[t] += float(w[t, j])
    bound = TOL * wsum[:, None] * colmax[None, :] + 2.0 ** -8 * np.abs(ref) + 1e-6
    err = np.abs(got - ref)
    assert (err <= bound).all(), f"worst error / bound {np.max(err / bound):.3f}"
    if drop:
        assert (wsum < 1 - 1e-6).any(), "the dropped block held no routed pair"


@pytest.mark.parametrize("case", COMBINE_CASES[:2], ids=[f"t{c[0]}e{c[1]}" for c in COMBINE_CASES[:2]])
def test_moe_combine_one_hot_weights_return_the_slot_row(case):
    """With weight 1 on slot j and 0 elsewhere, each token's output is its
    slot-j row byte for byte (one fma with 1, zero terms add nothing, and the
    rounding returns the bf16 value)."""
    tokens, experts, topk, block, k, widths, bits, cb = case
    layer, r, x = _setup(*case, seed=7400 + tokens)
    y, ids, be = _routed_rows(layer, r, x, tokens, topk, block, r.block_expert)
    ids_np = r.sorted_ids.numpy()
    for j in range(topk):
        w = torch.zeros((tokens, topk), dtype=torch.float32)
        w[:, j] = 1.0
        out = E.moe_combine(y, ids, be, block, experts, w.to(DEV), topk)
        torch.cuda.synchronize()
        rows = [int(np.nonzero(ids_np == t * topk + j)[0][0]) for t in range(tokens)]
        assert torch.equal(out.view(torch.int16), y[rows].view(torch.int16))


def test_moe_combine_scratch_needs_no_clearing():
    """Any contents of the pair-row table before the call (garbage, or rows of
    another routing) give the same bytes as a fresh table."""
    case = CASES[1]
    tokens, experts, topk, block, k, widths, bits, cb = case
    layer, r, x = _setup(*case, seed=7500)
    y, ids, be = _routed_rows(layer, r, x, tokens, topk, block, r.block_expert)
    w = synthetic.make_topk_weights(tokens, topk, seed=7501).to(DEV)
    want = E.moe_combine(y, ids, be, block, experts, w, topk)
    g = torch.Generator().manual_seed(7502)
    for lo, hi in ((-5, r.rows + 5), (0, r.rows)):
        junk = torch.randint(lo, hi, (tokens * topk,), generator=g, dtype=torch.int32).to(DEV)
        got = E.moe_combine(y, ids, be, block, experts, w, topk, pair_rows=junk)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    # a table left by another routing of the same tokens
    r2 = synthetic.make_routing(tokens, experts, topk, block, seed=7503)
    table = torch.empty(tokens * topk, dtype=torch.int32, device=DEV)
    E.moe_combine(y[:r2.rows] if r2.rows <= r.rows else y, r2.sorted_ids.to(DEV)[:min(r2.rows, r.rows)],
                  r2.block_expert.to(DEV)[:min(r2.rows, r.rows) // block], block, experts, w, topk,
                  pair_rows=table)
    got = E.moe_combine(y, ids, be, block, experts, w, topk, pair_rows=table)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
