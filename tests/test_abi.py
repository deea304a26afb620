"""C-ABI checks that need no GPU: the library loads, exports every declared
symbol, and rejects invalid calls on the host before launching anything."""
import ctypes
import os
import re

import pytest

from exl3_trellis_quantized_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "exl3.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(exl3_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    try:
        return B.lib()
    except ImportError as e:  # the build step must have run first
        pytest.fail(str(e))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert "exl3_gemm" in names and "exl3_input_transform" in names and "exl3_gemm_splitk" in names
    for name in names:
        assert hasattr(L, name), name


def test_status_strings(L):
    assert L.exl3_status_string(0) == b"ok"
    assert L.exl3_status_string(1) == b"invalid argument"
    assert L.exl3_status_string(3) == b"split-k workspace too small"


def test_splitk_policy_is_shape_only(L):
    # pure host function of (k, n)
    assert L.exl3_splitk_parts(17408, 5120) >= 2  # down_proj: 40 column blocks
    assert L.exl3_splitk_parts(5120, 154880) == 1  # lm_head fills the GPU
    assert L.exl3_splitk_parts(1024, 512) == 8  # capped at k/128
    assert L.exl3_splitk_parts(100, 128) == 0  # invalid shape
    for k, n in [(2048, 4096), (5120, 12288), (5120, 34816), (12288, 4096)]:
        p = L.exl3_splitk_parts(k, n)
        assert 1 <= p <= min(16, k // 128)
        assert L.exl3_splitk_workspace_bytes(9, k, n) == p * 9 * n * 4


FAKE = 1 << 20  # a 16-byte-aligned address; never dereferenced because validation fails first


def _gemm(L, m=4, k=256, bits=4, cb=1, n=256, cols=(0, 256), dtype=1, xh=FAKE, tr=FAKE, svh=FAKE, y=FAKE):
    arr = (ctypes.c_int32 * len(cols))(*cols)
    return L.exl3_gemm(ctypes.c_void_p(xh), m, k, ctypes.c_void_p(tr), bits, cb, ctypes.c_void_p(svh), arr,
                       len(cols) - 1, ctypes.c_void_p(y), dtype, n, None)


@pytest.mark.parametrize(
    "kw",
    [
        dict(m=-1),
        dict(k=200),
        dict(k=0),
        dict(n=384, cols=(0, 256)),
        dict(bits=0),
        dict(bits=9),
        dict(cb=3),
        dict(dtype=2),
        dict(cols=(0, 100, 256)),
        dict(cols=(0, 256, 256)),
        dict(cols=(128, 256)),
        dict(xh=0),
        dict(tr=FAKE + 8),
        dict(y=FAKE + 2),
    ],
)
def test_gemm_rejects_invalid_arguments(L, kw):
    assert _gemm(L, **kw) == 1


def test_empty_batch_is_a_no_op(L):
    assert _gemm(L, m=0) == 0
    assert _gemm(L, m=0, xh=0, y=0) == 0  # nothing is dereferenced
    assert _gemm(L, m=0, tr=0) == 1


def test_splitk_rejects_small_workspace(L):
    cols = (ctypes.c_int32 * 2)(0, 512)
    need = L.exl3_splitk_workspace_bytes(3, 1024, 512)
    st = L.exl3_gemm_splitk(ctypes.c_void_p(FAKE), 3, 1024, ctypes.c_void_p(FAKE), 2, 0, ctypes.c_void_p(FAKE), cols,
                            1, ctypes.c_void_p(FAKE), 0, 512, ctypes.c_void_p(FAKE), need - 4, None)
    assert st == 3


def _shape_call(L, shape, m, k, n, split=False):
    cols = (ctypes.c_int32 * 2)(0, n)
    v = ctypes.c_void_p(FAKE)
    acc = v if split else None
    nbytes = L.exl3_splitk_workspace_bytes(m, k, n) if split else 0
    return L.exl3_test_gemm_shape(shape, v, m, k, v, 4, 1, v, cols, 1, v, 1, n, acc, nbytes, None)


@pytest.mark.parametrize("shape,m,k,n,split", [
    (18, 8, 1024, 512, True),     # four-atom tensor-memory tiles on 128-row parts (P = 8 > k/256)
    (21, 8, 1024, 512, True),
    (28, 8, 1024, 512, True),
    (18, 33, 1024, 512, False),   # more rows than the shape holds
    (21, 17, 1024, 512, False),
    (28, 129, 1024, 512, False),
    (28, 64, 384, 512, False),    # odd k/128: no four-atom stages
    (8, 8, 1024, 4864, True),     # shared-memory four-atom tiles never run split-k parts, even 256-row ones
    (12, 8, 2048, 4096, True),
])
def test_tile_shape_support_rules(L, shape, m, k, n, split):
    """Host-side shape checks of exl3_test_gemm_shape: a shape that cannot run
    the call returns EXL3_EUNSUPPORTED before any launch (no GPU needed)."""
    if split:
        assert L.exl3_splitk_parts(k, n) > 1
    assert _shape_call(L, shape, m, k, n, split) == 2


def test_tile_shape_out_of_range(L):
    assert _shape_call(L, B.TEST_TILE_SHAPES, 8, 1024, 512) == 1
    assert _shape_call(L, -2, 8, 1024, 512) == 1


def test_input_transform_rejects_invalid(L):
    v = ctypes.c_void_p(FAKE)
    assert L.exl3_input_transform(v, 1, 4, 200, v, 1, v, None) == 1
    assert L.exl3_input_transform(v, 1, 4, 256, v, 0, v, None) == 1
    assert L.exl3_input_transform(v, 1, 4, 256, v, 9, v, None) == 1
    assert L.exl3_input_transform(ctypes.c_void_p(FAKE + 4), 1, 4, 256, v, 1, v, None) == 1
    assert L.exl3_input_transform(v, 1, 0, 256, v, 1, v, None) == 0


def test_swiglu_transform_rejects_invalid(L):
    v = ctypes.c_void_p(FAKE)
    assert L.exl3_input_transform_swiglu(v, 1, 4, 200, v, 1, v, None) == 1  # k not a multiple of 128
    assert L.exl3_input_transform_swiglu(v, 1, 4, 256, v, 0, v, None) == 1  # no shard
    assert L.exl3_input_transform_swiglu(v, 2, 4, 256, v, 1, v, None) == 1  # dtype
    assert L.exl3_input_transform_swiglu(ctypes.c_void_p(FAKE + 4), 1, 4, 256, v, 1, v, None) == 1
    assert L.exl3_input_transform_swiglu(v, 1, 0, 256, v, 1, v, None) == 0  # empty batch


def test_moe_entry_points_reject_invalid(L):
    v = ctypes.c_void_p(FAKE)
    cols = (ctypes.c_int32 * 2)(0, 256)
    # block 64 / rows not a multiple of the block / no experts
    assert L.exl3_moe_input_transform(v, 1, 4, 256, v, 64, 2, v, 64, v, 1, 4, v, None) == 1
    assert L.exl3_moe_input_transform(v, 1, 4, 256, v, 40, 2, v, 32, v, 1, 4, v, None) == 1
    assert L.exl3_moe_input_transform(v, 1, 4, 256, v, 64, 2, v, 32, v, 1, 0, v, None) == 1
    assert L.exl3_moe_input_transform(v, 1, 4, 256, v, 0, 2, v, 32, v, 1, 4, v, None) == 0  # nothing routed
    assert L.exl3_moe_gemm(v, 64, 256, v, 4, 1, v, cols, 1, v, 64, 4, v, 1, 256, None) == 1
    assert L.exl3_moe_gemm(v, 40, 256, v, 4, 1, v, cols, 1, v, 32, 4, v, 1, 256, None) == 1
    assert L.exl3_moe_gemm(v, 64, 256, v, 4, 1, v, cols, 1, None, 32, 4, v, 1, 256, None) == 1  # no block ids
    assert L.exl3_moe_gemm(v, 0, 256, v, 4, 1, v, cols, 1, v, 32, 4, v, 1, 256, None) == 0
    # 16-row blocks are accepted (empty batches, so nothing launches)
    assert L.exl3_moe_input_transform(v, 1, 4, 256, v, 0, 2, v, 16, v, 1, 4, v, None) == 0
    assert L.exl3_moe_gemm(v, 0, 256, v, 4, 1, v, cols, 1, v, 16, 4, v, 1, 256, None) == 0
    assert L.exl3_moe_gemm(v, 24, 256, v, 4, 1, v, cols, 1, v, 16, 4, v, 1, 256, None) == 1  # 24 rows: not whole blocks


def test_moe_combine_rejects_invalid(L):
    v = ctypes.c_void_p(FAKE)
    odd = ctypes.c_void_p(FAKE + 4)

    def call(y=v, rows=64, n=256, block=32, experts=4, w=v, tokens=8, topk=2, pair_rows=v, out=v, out_dtype=1):
        return L.exl3_moe_combine(y, 1, rows, n, v, v, block, experts, w, tokens, topk, pair_rows, out, out_dtype,
                                  None)

    assert call(block=64) == 1  # block size
    assert call(rows=40) == 1  # rows not whole blocks
    assert call(n=200) == 1  # n not a multiple of 128
    assert call(topk=0) == 1 and call(topk=65) == 1
    assert call(experts=0) == 1
    assert call(out_dtype=2) == 1
    assert call(pair_rows=None) == 1  # no scratch table
    assert call(w=None) == 1  # no weights
    assert call(out=odd) == 1 and call(y=odd) == 1  # misaligned
    assert call(tokens=0, pair_rows=None, out=None, w=None) == 0  # no tokens: nothing to do


def test_test_entry_points_reject_invalid(L):
    v = ctypes.c_void_p(FAKE)
    assert L.exl3_test_wait_timeout(None, None) == 1
    assert L.exl3_test_wait_timeout(ctypes.c_void_p(FAKE + 2), None) == 1  # misaligned
    assert L.exl3_test_codebook(7, v, None) == 1
    assert L.exl3_test_unpack(v, 9, 0, 64, 64, v, None) == 1
    assert L.exl3_test_unpack(v, 3, 0, 40, 64, v, None) == 1


def test_autotune_switch(L):
    """The tuner's switch and cache are host state: no device call is made."""
    assert L.exl3_set_autotune(2) == 1  # EXL3_EINVAL
    assert L.exl3_set_autotune(-1) == 1
    assert L.exl3_set_autotune(1) == 0
    assert L.exl3_set_autotune(0) == 0
    assert L.exl3_clear_autotune() == 0
    assert L.exl3_autotune_entries() == 0
