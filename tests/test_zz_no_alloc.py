"""The split-k GEMM for callers that cannot allocate (exl3_gemm_splitk_noalloc).

Callers such as a plugin living inside a host program that owns every device
allocation cannot hand the library a workspace.  This entry point keeps its
fp32 partials in a scratch array built into the library instead.  These tests
call it through the C ABI and check that it gives the same result as
exl3_gemm_splitk with a caller-supplied workspace, on three calls in a row
(the second smaller, so anything the first left in the shared array would
show, the third at the first call's batch again), that a warmed-up call takes
no device memory (free bytes before and after it are equal), and that a batch
too large for the array is refused without a launch.

This file is named to be collected last.
"""
import os
import re

import numpy as np
import pytest
import torch

import exl3_trellis_quantized_gb300 as E
from exl3_trellis_quantized_gb300 import binding as B
from exl3_trellis_quantized_gb300 import synthetic

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL = 4e-3  # per output column, relative to the column's largest magnitude (as in the parity tests)
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_limit():
    with open(os.path.join(ROOT, "include", "exl3.h")) as f:
        text = f.read()
    mt = re.search(r"#define EXL3_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    return int(mt.group(1)) << int(mt.group(2))


def test_binding_limit_matches_header():
    assert B.NOALLOC_SCRATCH_BYTES == _header_limit()


def test_noalloc_matches_splitk_on_two_calls():
    k, n, bits, cb = 1024, 512, 3, 1
    assert E.splitk_parts(k, n) > 1  # the split-k parts really use the scratch
    layer = synthetic.make_layer(k, [n], bits, cb, seed=321)
    tr, suh, svh = layer.trellis.to(DEV), layer.suh.to(DEV), layer.svh.to(DEV)
    first = None
    for m, seed in ((40, 5), (7, 6), (40, 5)):
        x = synthetic.make_x(m, k, seed=seed).to(DEV)
        xh = E.input_transform(x, suh)
        acc = torch.zeros(E.splitk_workspace_bytes(m, k, n) // 4, dtype=torch.float32, device=DEV)
        want = E.gemm_splitk(xh, tr, bits, cb, svh, layer.shard_cols, acc)
        got = B.gemm_splitk_noalloc(xh, tr, bits, cb, svh, layer.shard_cols)
        torch.cuda.synchronize()
        w = want.float().cpu().numpy()
        g = got.float().cpu().numpy()
        colmax = np.abs(w).max(axis=0)
        assert np.all(np.abs(g - w) <= TOL * colmax), f"m={m}: outside tolerance"
        # the same kernels run in the same order, so the bytes agree as well
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"m={m}: bytes differ"
        if first is None:
            first = got.clone()
    # the third call repeats the first after a smaller one used the array
    assert torch.equal(got.view(torch.int16), first.view(torch.int16))
    assert E.device_status() == 0


def test_noalloc_call_takes_no_device_memory():
    k, n, bits, cb, m = 2048, 256, 4, 0, 64
    assert E.splitk_parts(k, n) > 1
    layer = synthetic.make_layer(k, [n], bits, cb, seed=323)
    tr, suh, svh = layer.trellis.to(DEV), layer.suh.to(DEV), layer.svh.to(DEV)
    xh = E.input_transform(synthetic.make_x(m, k, seed=7).to(DEV), suh)
    y = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
    B.gemm_splitk_noalloc(xh, tr, bits, cb, svh, layer.shard_cols, out=y)  # loads the kernels
    torch.cuda.synchronize()
    want = y.clone()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        B.gemm_splitk_noalloc(xh, tr, bits, cb, svh, layer.shard_cols, out=y)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free bytes moved by {free0 - free1} over three calls"
    assert torch.equal(y.view(torch.int16), want.view(torch.int16))
    assert E.device_status() == 0


def test_noalloc_refuses_batch_beyond_scratch():
    k, n, bits, cb = 1024, 512, 3, 1
    layer = synthetic.make_layer(k, [n], bits, cb, seed=322)
    m = 1
    while E.splitk_workspace_bytes(m, k, n) <= B.NOALLOC_SCRATCH_BYTES:
        m *= 2
    xh = torch.zeros((1, m, k), dtype=torch.float16, device=DEV)
    y = torch.full((m, n), 7.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(E.Exl3Error, match="scratch"):
        B.gemm_splitk_noalloc(xh, layer.trellis.to(DEV), bits, cb, layer.svh.to(DEV), layer.shard_cols, out=y)
    torch.cuda.synchronize()
    assert bool((y == 7.0).all()), "a refused call must launch nothing"
