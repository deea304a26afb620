"""GPU parity: the CUDA path through the C ABI against the FP64 oracle.

Bars (from the layer's specification):
  * codebook values and unpacked Wq: bit-exact;
  * input rotation: within one fp16 rounding of the exact value plus the fp32
    butterfly's rounding bound;
  * linear output: |y_gpu - y_oracle| <= 4e-3 * max_r |y_oracle[r, c]| per column,
    the max taken over the rows of the largest batch of the case;
  * every row byte-equal at every batch size; a fused multi-shard launch
    byte-equal to separate launches; the split-k workspace zero after a call.
"""
import numpy as np
import pytest
import torch

import exl3_trellis_quantized_gb300 as E
from exl3_trellis_quantized_gb300 import binding as B
from exl3_trellis_quantized_gb300 import synthetic
from oracle import exl3_oracle as O
from oracle_check import TOL, assert_columns

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _no_device_errors():
    """Every test must leave no wait-timeout flag behind."""
    yield
    assert E.device_status() == 0, "a kernel gave up on a bounded wait"


def _np(t):
    return t.detach().float().cpu().numpy()


def _bits(t):
    return t.detach().cpu().numpy().view(np.uint16)


def _dev(layer):
    return (layer.trellis.to(DEV), layer.suh.to(DEV), layer.svh.to(DEV))


def _oracle(x, layer, col_blocks=None):
    return O.linear(_np(x), layer.trellis.numpy(), layer.bits, layer.codebook, _np(layer.suh), _np(layer.svh),
                    layer.shard_cols, col_blocks=col_blocks)


_assert_columns = assert_columns


def _run(layer, x, out_dtype, split, m=None):
    tr, suh, svh = _dev(layer)
    xd = x.to(DEV) if m is None else x[:m].to(DEV)
    acc = None
    if split:
        nbytes = E.splitk_workspace_bytes(xd.shape[0], layer.k, layer.n)
        acc = torch.zeros(max(1, nbytes // 4), dtype=torch.float32, device=DEV)
    y = E.linear(xd, tr, layer.bits, layer.codebook, suh, svh, layer.shard_cols, out_dtype=out_dtype, acc=acc)
    torch.cuda.synchronize()
    return y, acc


# ---------------------------------------------------------------------------
# decode primitives
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("cb", [0, 1, 2])
def test_codebook_all_states_bit_exact(cb):
    got = _bits(E.binding.test_codebook(cb, DEV))
    want = O.codebook(cb, np.arange(65536))
    assert np.array_equal(got, want), f"{np.sum(got != want)} states differ"


@pytest.mark.parametrize("bits", range(1, 9))
@pytest.mark.parametrize("cb", [0, 1, 2])
def test_unpack_bit_exact(bits, cb):
    g = torch.Generator().manual_seed(40 + 3 * bits + cb)
    tr = synthetic.random_trellis(64, 96, bits, g)
    got = _bits(E.binding.test_unpack(tr.to(DEV), bits, cb))
    want = O.f64_to_half_bits(O.dequantize(tr.numpy(), bits, cb))
    assert np.array_equal(got, want)


# ---------------------------------------------------------------------------
# input rotation
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("xdtype", [torch.bfloat16, torch.float16])
def test_input_transform_parity(xdtype):
    m, k, s = 37, 640, 3
    layer = synthetic.make_layer(k, [128] * s, 4, 1, seed=5)
    x = synthetic.make_x(m, k, seed=5).to(xdtype)
    xh = E.input_transform(x.to(DEV), layer.suh.to(DEV))
    torch.cuda.synchronize()
    got = _np(xh)
    ref = O.input_transform(_np(x), _np(layer.suh))
    # fp32 butterfly: 7 rounded add stages over 128 exact products
    xs = np.abs(_np(x))[None] * np.abs(_np(layer.suh))[:, None, :]
    blk_sum = np.repeat(xs.reshape(s, m, k // 128, 128).sum(-1), 128, axis=-1)
    e = 8 * 2.0 ** -24 * blk_sum * 2.0 ** -4
    # rounding to fp16 is monotonic: the result lies between the roundings of ref -+ e
    lo = (ref - e).astype(np.float16).astype(np.float64)
    hi = (ref + e).astype(np.float16).astype(np.float64)
    bad = (got < lo) | (got > hi)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{bad.sum()} bad; first {tuple(i)}: got {got[tuple(i)]!r} ref {ref[tuple(i)]!r} "
                             f"lo {lo[tuple(i)]!r} hi {hi[tuple(i)]!r}")


def _fp32_butterfly_fp16(x, suh):
    """x * suh, the 128-point butterfly in fp32 (strides 1, 2, ..., 64, each
    stage (a, b) -> (a + b, a - b) rounded to nearest even), times 2^-4, then
    fp16 round-to-nearest-even: the transform's arithmetic written out with
    numpy's IEEE float32, for a bit-level check of the kernels."""
    s, k = suh.shape
    m = x.shape[0]
    v = (x.astype(np.float32)[None] * suh.astype(np.float32)[:, None, :]).reshape(s, m, k // 128, 128)
    idx = np.arange(128)
    st = 1
    while st < 128:
        lo = idx[(idx & st) == 0]
        a, b = v[..., lo].copy(), v[..., lo + st].copy()
        v[..., lo] = a + b
        v[..., lo + st] = a - b
        st <<= 1
    return (v.reshape(s, m, k) * np.float32(0.0625)).astype(np.float16)


@pytest.mark.parametrize("xdtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("m,k,s", [(37, 640, 3), (1, 128, 1), (300, 5120, 2)])
def test_input_transform_bits_equal_fp32_butterfly(xdtype, m, k, s):
    """The transform's fp16 bytes equal the fixed-order fp32 butterfly written
    out on the host (x * suh is exact in fp32, every stage rounds once, in the
    stride order 1..64), for the plain and the gathered transform (one expert,
    identity routing; padding rows zero)."""
    g = torch.Generator().manual_seed(70 + m)
    suh = (torch.rand(s, k, generator=g) * 0.4 + 0.8).to(torch.float16)
    suh[:, ::5] = -suh[:, ::5]
    x = synthetic.make_x(m, k, seed=71).to(xdtype)
    want = _fp32_butterfly_fp16(x.float().numpy(), suh.float().numpy())
    plain = E.input_transform(x.to(DEV), suh.to(DEV))
    assert np.array_equal(plain.cpu().numpy().view(np.int16), want.view(np.int16))
    block = 16
    rows = (m + block - 1) // block * block
    ids = torch.arange(rows, dtype=torch.int32)
    ids[m:] = m  # padding rows (an id past the last pair)
    grouped = E.moe_input_transform(x.to(DEV), ids.to(DEV), 1, torch.zeros(rows // block, dtype=torch.int32,
                                    device=DEV), block, suh[None].to(DEV))
    got = grouped.cpu().numpy()
    assert np.array_equal(got[:, :m].view(np.int16), want.view(np.int16))
    assert not got[:, m:].any()


@pytest.mark.parametrize("xdtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("m,k,s", [(37, 640, 3), (1, 128, 1), (300, 5120, 2)])
def test_input_transform_bits_equal_gathered_form(xdtype, m, k, s):
    """The plain transform and the grouped-expert (gathered) transform run the
    butterfly's stages in the same stride order on the same pairs, so with one
    expert and the identity routing their fp16 bytes are equal for every row
    and shard."""
    g = torch.Generator().manual_seed(60 + m)
    suh = (torch.rand(s, k, generator=g) * 0.4 + 0.8).to(torch.float16)
    suh[:, ::3] = -suh[:, ::3]
    x = synthetic.make_x(m, k, seed=61).to(xdtype).to(DEV)
    plain = E.input_transform(x, suh.to(DEV))
    block = 16
    rows = (m + block - 1) // block * block
    ids = torch.arange(rows, dtype=torch.int32)
    ids[m:] = m  # padding rows (an id past the last pair)
    grouped = E.moe_input_transform(x, ids.to(DEV), 1, torch.zeros(rows // block, dtype=torch.int32, device=DEV), block,
                                    suh[None].to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(plain.view(torch.int16), grouped[:, :m].contiguous().view(torch.int16))


# ---------------------------------------------------------------------------
# the layer: coverage of widths x codebooks, batch sizes, dtypes
# ---------------------------------------------------------------------------

M_SET = [1, 2, 7, 16, 64, 300]


@pytest.mark.parametrize("bits", range(1, 9))
@pytest.mark.parametrize("cb", [0, 1, 2])
def test_linear_coverage_small_split(bits, cb):
    """K=1024, N=512 (under 96 column blocks, exercising split-k), all rows checked."""
    k, n = 1024, 512
    layer = synthetic.make_layer(k, [n], bits, cb, seed=1001 + 10 * bits + cb)
    x = synthetic.make_x(300, k, seed=1001)
    out_dtype = torch.float16 if (bits + cb) % 2 else torch.bfloat16
    ref = _oracle(x, layer)
    for split in (False, True):
        y, acc = _run(layer, x, out_dtype, split)
        _assert_columns(_np(y), ref, f"split={split}")
        if split:
            assert not acc.any(), "split-k workspace not re-zeroed"
        for m in M_SET[:-1]:
            ym, _ = _run(layer, x, out_dtype, split, m=m)
            assert torch.equal(ym.view(torch.int16), y[:m].view(torch.int16)), f"row bytes differ at m={m}"


@pytest.mark.parametrize("bits", range(1, 9))
@pytest.mark.parametrize("cb", [0, 1, 2])
def test_linear_coverage_2048(bits, cb):
    """K=2048, N=2048; three sampled column blocks checked against the oracle."""
    k, n = 2048, 2048
    layer = synthetic.make_layer(k, [n], bits, cb, seed=1001 + 10 * bits + cb + 5)
    x = synthetic.make_x(300, k, seed=1002)
    out_dtype = torch.bfloat16 if (bits + cb) % 2 else torch.float16
    blocks = [0, 7, 15]
    ref = _oracle(x, layer, blocks)
    y, _ = _run(layer, x, out_dtype, False)
    got = _np(y).reshape(300, 16, 128)[:, blocks].reshape(300, -1)
    _assert_columns(got, ref)
    for m in (1, 16, 64):
        ym, _ = _run(layer, x, out_dtype, False, m=m)
        assert torch.equal(ym.view(torch.int16), y[:m].view(torch.int16))


SHAPE_CASES = [
    # k, n, bits, codebook, batch sizes: chosen so the kernel switches tile shapes
    # (128-column small-batch CTAs, 32/64-column cluster strips, one and two row
    # groups, 128 and 256 columns) between the batch sizes of one case
    (1024, 12288, 4, 0, [3, 16, 77, 300]),
    (1024, 640, 3, 2, [5, 40, 300]),
    (384, 4096, 5, 1, [2, 20, 150]),  # an odd number of 128-blocks of k
    (2048, 2048, 6, 1, [1, 33, 129, 257]),
]


@pytest.mark.parametrize("k,n,bits,cb,ms", SHAPE_CASES, ids=[f"{c[0]}x{c[1]}" for c in SHAPE_CASES])
def test_rows_byte_equal_across_tile_shapes(k, n, bits, cb, ms):
    layer = synthetic.make_layer(k, [n], bits, cb, seed=3000 + n)
    x = synthetic.make_x(max(ms), k, seed=3000)
    y, _ = _run(layer, x, torch.bfloat16, False)
    for m in ms[:-1]:
        ym, _ = _run(layer, x, torch.bfloat16, False, m=m)
        assert torch.equal(ym.view(torch.int16), y[:m].view(torch.int16)), f"row bytes differ at m={m}"
    blocks = [0, n // 128 - 1]
    ref = _oracle(x, layer, blocks)
    got = _np(y).reshape(max(ms), n // 128, 128)[:, blocks].reshape(max(ms), -1)
    _assert_columns(got, ref)


TILE_CASES = [
    # k, shard widths, bits, codebook: every tile shape against the library's choice
    (1024, [512], 3, 1),
    (2048, [256, 256], 6, 2),
    (1152, [384, 128], 2, 0),  # an odd number of 128-blocks of k; 128-aligned shard edges
    (1024, [1024], 8, 1),
    (2048, [384, 384], 4, 2),  # 384-aligned edges: 96-column strips over two shards
]


@pytest.mark.parametrize("k,widths,bits,cb", TILE_CASES,
                         ids=[f"{c[0]}x{sum(c[1])}b{c[2]}cb{c[3]}" for c in TILE_CASES])
@pytest.mark.parametrize("split", [False, True], ids=["gemm", "splitk"])
def test_every_tile_shape_byte_equal(k, widths, bits, cb, split):
    """Each tile shape computes every element with the same k16 steps in the same
    order, so all of them give the bytes of the library's own choice (and the
    split-k workspace is left zeroed by each)."""
    layer = synthetic.make_layer(k, widths, bits, cb, seed=4100 + k + bits)
    tr, suh, svh = _dev(layer)
    n = layer.n
    ran = set()
    for m in (5, 32, 300, 700):
        x = synthetic.make_x(m, k, seed=4200 + m).to(DEV)
        xh = E.input_transform(x, suh)
        acc = (torch.zeros(max(1, E.splitk_workspace_bytes(m, k, n) // 4), dtype=torch.float32, device=DEV)
               if split else None)
        want = (E.gemm_splitk(xh, tr, bits, cb, svh, layer.shard_cols, acc) if split
                else E.gemm(xh, tr, bits, cb, svh, layer.shard_cols))
        for shape in range(B.TEST_TILE_SHAPES):
            got = B.test_gemm_shape(shape, xh, tr, bits, cb, svh, layer.shard_cols, acc)
            if got is None:
                continue
            ran.add(shape)
            assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"shape {shape} m={m}: bytes differ"
            if split:
                assert bool((acc == 0).all()), f"shape {shape} m={m}: workspace not re-zeroed"
    # the cases reach every shape that their sizes allow
    need = {1, 2, 3, 4, 6, 19, 23, 25, 26} | ({5, 7} if all(w % 256 == 0 for w in widths) else set())
    need |= {10, 11} if all(w % 384 == 0 for w in widths) else set()
    if not split and (k // 128) % 2 == 0:
        need |= {0, 8, 13, 15, 16, 17, 18, 21, 24, 28} | ({9, 14, 20, 22, 27} if all(w % 384 == 0 for w in widths) else set())
    if not split and k % 512 == 0:
        need |= {12}
    assert need <= ran, f"shapes not exercised: {sorted(need - ran)}"


TM_SHAPES = {18: 32, 19: 32, 21: 16, 23: 16, 24: 64, 25: 64, 26: 128, 28: 128}  # tensor-memory shapes and their rows


@pytest.mark.parametrize("bits", range(1, 9))
@pytest.mark.parametrize("cb", [0, 1, 2])
def test_tensor_memory_shapes_every_width(bits, cb):
    """The tensor-memory kernel's column decode (16 values of one column a
    lane) at every width and codebook: each of its shapes gives the bytes of
    the shared-memory kernel's tiles (64-column strips, shape 1, up to 32 rows;
    128 x 128 tiles, shape 3, above; their decode takes 8 consecutive values a
    lane), plain and split-k, and meets the oracle."""
    k, n = 512, 256
    layer = synthetic.make_layer(k, [n], bits, cb, seed=4500 + 3 * bits + cb)
    tr, suh, svh = _dev(layer)
    x = synthetic.make_x(128, k, seed=4501)
    ref = _oracle(x, layer)
    for m in (1, 7, 16, 32, 50, 64, 100, 128):
        xh = E.input_transform(x[:m].to(DEV), suh)
        ref_shape = 1 if m <= 32 else 3
        want = B.test_gemm_shape(ref_shape, xh, tr, bits, cb, svh, layer.shard_cols)
        assert torch.equal(E.gemm(xh, tr, bits, cb, svh, layer.shard_cols).view(torch.int16), want.view(torch.int16))
        acc = torch.zeros(max(1, E.splitk_workspace_bytes(m, k, n) // 4), dtype=torch.float32, device=DEV)
        want_split = B.test_gemm_shape(ref_shape, xh, tr, bits, cb, svh, layer.shard_cols, acc)
        assert want_split is not None
        for shape, rows in TM_SHAPES.items():
            if m > rows:
                continue
            got = B.test_gemm_shape(shape, xh, tr, bits, cb, svh, layer.shard_cols)
            assert got is not None, f"shape {shape} refused m={m}"
            assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"shape {shape} m={m}: bytes differ"
            if shape in (19, 23, 25, 26):  # the two-atom shapes also run split-k parts
                got = B.test_gemm_shape(shape, xh, tr, bits, cb, svh, layer.shard_cols, acc)
                assert got is not None
                assert torch.equal(got.view(torch.int16), want_split.view(torch.int16)), f"split shape {shape} m={m}"
                assert not bool(acc.any())
        _assert_columns(_np(want), ref[:m], f"bits={bits} cb={cb} m={m}", ref_batch=ref)


def test_splitk_one_part_is_gemm():
    """A layer whose column blocks fill the GPU gets one part: the split-k call
    then gives exl3_gemm's bytes and leaves the workspace as it found it (here
    NaN-filled)."""
    k, n, bits, cb = 256, 152 * 128, 4, 1
    assert E.splitk_parts(k, n) == 1
    layer = synthetic.make_layer(k, [n], bits, cb, seed=4800)
    tr, suh, svh = _dev(layer)
    for m in (1, 16, 100):
        xh = E.input_transform(synthetic.make_x(m, k, seed=4801).to(DEV), suh)
        want = E.gemm(xh, tr, bits, cb, svh, layer.shard_cols)
        acc = torch.full((E.splitk_workspace_bytes(m, k, n) // 4,), float("nan"), dtype=torch.float32, device=DEV)
        got = E.gemm_splitk(xh, tr, bits, cb, svh, layer.shard_cols, acc)
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"m={m}"
        assert bool(torch.isnan(acc).all()), f"m={m}: workspace touched"


@pytest.mark.parametrize("bits", [1, 3, 4, 6, 8])
@pytest.mark.parametrize("cb", [0, 1, 2])
def test_split_four_atom_parts(bits, cb):
    """Split-k parts of whole 256-row units of k (k/128 even and P <= k/256:
    here 1024 x 4864, 38 column blocks, P = 4): the tensor-memory kernel's
    four-atom shapes run them and give the bytes of the shared-memory tiles'
    parts and of its two-atom shapes, the workspace comes back zeroed, and the
    result meets the oracle on a first, a middle and the last column block."""
    k, n = 1024, 4864
    assert E.splitk_parts(k, n) == 4
    layer = synthetic.make_layer(k, [n], bits, cb, seed=4700 + 3 * bits + cb)
    tr, suh, svh = _dev(layer)
    x = synthetic.make_x(64, k, seed=4701)
    blocks = [0, 17, 37]
    ref = _oracle(x, layer, col_blocks=blocks)
    cols = np.concatenate([np.arange(128 * b, 128 * b + 128) for b in blocks])
    for m in (1, 7, 16, 29, 32, 50, 64):
        xh = E.input_transform(x[:m].to(DEV), suh)
        acc = torch.zeros(max(1, E.splitk_workspace_bytes(m, k, n) // 4), dtype=torch.float32, device=DEV)
        want = B.test_gemm_shape(1 if m <= 32 else 3, xh, tr, bits, cb, svh, layer.shard_cols, acc)
        assert want is not None
        want = want.clone()
        got = E.gemm_splitk(xh, tr, bits, cb, svh, layer.shard_cols, acc)
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"m={m}: planned split differs"
        for shape, rows in TM_SHAPES.items():
            if m > rows:
                continue
            got = B.test_gemm_shape(shape, xh, tr, bits, cb, svh, layer.shard_cols, acc)
            assert got is not None, f"shape {shape} refused m={m}"
            assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"shape {shape} m={m}: bytes differ"
            assert not bool(acc.any()), f"shape {shape} m={m}: workspace not re-zeroed"
        _assert_columns(_np(want)[:, cols], ref[:m], f"bits={bits} cb={cb} m={m}", ref_batch=ref)


@pytest.mark.parametrize("m", [3, 16, 29, 61, 100])
def test_tensor_memory_kernel_many_items(m):
    """A persistent launch with several waves of work items and a ragged last
    wave (400 column blocks over the SMs), at ragged batch sizes: bytes of the
    column strips' launch, and the oracle on blocks of the first, a middle and
    the last wave."""
    k, n, bits, cb = 256, 400 * 128, 5, 1
    layer = synthetic.make_layer(k, [n], bits, cb, seed=4600)
    tr, suh, svh = _dev(layer)
    x = synthetic.make_x(128, k, seed=4601)
    xh = E.input_transform(x[:m].to(DEV), suh)
    shape = 23 if m <= 16 else 19 if m <= 32 else 24 if m <= 64 else 26
    got = B.test_gemm_shape(shape, xh, tr, bits, cb, svh, layer.shard_cols)
    strips = B.test_gemm_shape(3, xh, tr, bits, cb, svh, layer.shard_cols)  # 128 x 128 tiles, one per block
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), strips.view(torch.int16))
    blocks = [0, 151, 152, 303, 304, 399]
    ref = _oracle(x, layer, blocks)
    out = _np(got).reshape(m, n // 128, 128)[:, blocks].reshape(m, -1)
    _assert_columns(out, ref[:m], f"m={m}", ref_batch=ref)


def test_tile_shape_rejections():
    layer = synthetic.make_layer(1024, [384], 3, 1, seed=4300)
    tr, suh, svh = _dev(layer)
    x = synthetic.make_x(40, 1024, seed=4301).to(DEV)
    xh = E.input_transform(x, suh)
    assert B.test_gemm_shape(2, xh, tr, 3, 1, svh, layer.shard_cols) is None  # 40 rows > 32
    assert B.test_gemm_shape(5, xh, tr, 3, 1, svh, layer.shard_cols) is None  # 384 columns: not 256-aligned
    with pytest.raises(E.Exl3Error):  # past the last shape
        B.test_gemm_shape(B.TEST_TILE_SHAPES, xh, tr, 3, 1, svh, layer.shard_cols)


def test_fused_shards_equal_separate_launches():
    k, bits, cb = 512, 5, 2
    layer = synthetic.make_layer(k, [256, 128, 384], bits, cb, seed=77)
    x = synthetic.make_x(20, k, seed=77)
    y, _ = _run(layer, x, torch.bfloat16, False)
    tr, suh, svh = _dev(layer)
    xd = x.to(DEV)
    for s in range(3):
        a, b = layer.shard_cols[s], layer.shard_cols[s + 1]
        ys = E.linear(xd, tr[:, a // 16:b // 16].contiguous(), bits, cb, suh[s:s + 1].contiguous(),
                      svh[a:b].contiguous(), [0, b - a])
        torch.cuda.synchronize()
        assert torch.equal(ys.view(torch.int16), y[:, a:b].view(torch.int16)), s
    _assert_columns(_np(y), _oracle(x, layer))


def test_splitk_workspace_reused_across_calls():
    """One workspace, several calls on one stream: zero after each, results stable."""
    k, n, bits, cb = 1024, 512, 3, 1
    layer = synthetic.make_layer(k, [n], bits, cb, seed=88)
    x = synthetic.make_x(33, k, seed=88).to(DEV)
    tr, suh, svh = _dev(layer)
    acc = torch.zeros(E.splitk_workspace_bytes(33, k, n) // 4, dtype=torch.float32, device=DEV)
    ys = [E.linear(x, tr, bits, cb, suh, svh, layer.shard_cols, acc=acc) for _ in range(3)]
    torch.cuda.synchronize()
    assert not acc.any()
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))
    assert torch.equal(ys[0].view(torch.int16), ys[2].view(torch.int16))


def test_empty_batch():
    layer = synthetic.make_layer(256, [256], 4, 1, seed=3)
    tr, suh, svh = _dev(layer)
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    y = E.linear(x, tr, 4, 1, suh, svh, layer.shard_cols)
    assert y.shape == (0, 256)


# ---------------------------------------------------------------------------
# full-size layers, in the launch configuration the benchmark times; every row
# of sampled 128-column blocks is checked against the oracle
# ---------------------------------------------------------------------------

FULL = [
    # name, k, shard widths, bits, codebook, m, split: every layer at the batch
    # sizes the benchmark times it at (m = 1 is covered by the byte-equality
    # test below, whose rows equal those of the checked batches)
    ("single_2048x4096_4b_mcg_m16", 2048, [4096], 4, 1, 16, False),
    ("q_proj_5120x12288_6b_mcg_m16", 5120, [12288], 6, 1, 16, False),
    ("q_proj_5120x12288_6b_mcg_m512", 5120, [12288], 6, 1, 512, False),
    ("q_proj_5120x12288_6b_mcg_m4096", 5120, [12288], 6, 1, 4096, False),
    ("gate_up_5120x2x17408_5b_mul1_m16", 5120, [17408, 17408], 5, 2, 16, False),
    ("gate_up_5120x2x17408_5b_mul1_m512", 5120, [17408, 17408], 5, 2, 512, False),
    ("down_17408x5120_6b_mul1_splitk_m16", 17408, [5120], 6, 2, 16, True),
    ("down_17408x5120_6b_mul1_splitk_m512", 17408, [5120], 6, 2, 512, True),
    ("lm_head_4096x154880_6b_3inst_m16", 4096, [154880], 6, 0, 16, False),
    ("lm_head_4096x154880_6b_3inst_m512", 4096, [154880], 6, 0, 512, False),
    ("lm_head_4096x154880_6b_3inst_m2048", 4096, [154880], 6, 0, 2048, False),
    ("proj_12288x4096_5b_mcg_m16", 12288, [4096], 5, 1, 16, False),
    ("proj_12288x4096_5b_mcg_m512", 12288, [4096], 5, 1, 512, False),
    ("proj_12288x4096_5b_mcg_m2048", 12288, [4096], 5, 1, 2048, False),
]


def _sampled_blocks(layer):
    nb = layer.n // 128
    blocks = {0, nb // 2, nb - 1}
    for s in range(1, len(layer.shard_cols) - 1):  # first block of every further shard
        blocks.add(layer.shard_cols[s] // 128)
    return sorted(blocks)


@pytest.mark.parametrize("name,k,widths,bits,cb,m,split", FULL, ids=[f[0] for f in FULL])
def test_full_size_sampled(name, k, widths, bits, cb, m, split):
    """Every row of sampled 128-column blocks against the oracle, at full size."""
    layer = synthetic.make_layer(k, widths, bits, cb, seed=2000 + k + len(widths))
    x = synthetic.make_x(m, k, seed=2000)
    y, acc = _run(layer, x, torch.bfloat16, split)
    blocks = _sampled_blocks(layer)
    nb = layer.n // 128
    ref = _oracle(x, layer, blocks)  # the column max of the tolerance is over every row of the batch
    got = _np(y.view(m, nb, 128)[:, blocks].reshape(m, -1))
    _assert_columns(got, ref, name)
    assert not torch.isnan(y.float()).any()
    if split:
        assert not acc.any()


BENCH_SETS = [
    # name, k, shard widths, bits, codebook, split, the benchmark's batch sizes
    ("q_proj", 5120, [12288], 6, 1, False, [1, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096]),
    ("gate_up", 5120, [17408, 17408], 5, 2, False, [1, 16, 128, 512]),
    ("down_splitk", 17408, [5120], 6, 2, True, [1, 16, 128, 512]),
    ("lm_head", 4096, [154880], 6, 0, False, [1, 16, 512, 2048]),
    ("proj_12288x4096", 12288, [4096], 5, 1, False, [1, 16, 512, 2048]),
    ("single_2048x4096", 2048, [4096], 4, 1, False, [1, 16]),
]


@pytest.mark.parametrize("name,k,widths,bits,cb,split,ms", BENCH_SETS, ids=[b[0] for b in BENCH_SETS])
def test_full_size_rows_byte_equal_across_bench_batches(name, k, widths, bits, cb, split, ms):
    """Each row's output bytes do not depend on the batch it is computed in:
    the first m rows of the largest benchmarked batch equal a launch of those m
    rows alone, for every batch size the benchmark times the layer at (each one
    takes its own tile plan)."""
    layer = synthetic.make_layer(k, widths, bits, cb, seed=2100 + k)
    x = synthetic.make_x(max(ms), k, seed=2101)
    big, _ = _run(layer, x, torch.bfloat16, split)
    for m in ms[:-1]:
        y, acc = _run(layer, x, torch.bfloat16, split, m=m)
        assert torch.equal(y.view(torch.int16), big[:m].view(torch.int16)), f"{name}: rows differ at m={m}"
        if split:
            assert not acc.any()


SPLIT_CASES = [
    # k, shard widths, bits, codebook, m: pair launches whose partial last wave
    # is split off into a second launch of smaller tiles on 152 SMs
    (256, [12288], 4, 1, 1024),  # 192 pair CTAs: 40 of them become 40 pairs of 256-row x 128-column tiles
    (256, [10240, 2048], 3, 0, 1024),  # the split-off columns span both shards
    (256, [6144, 6144], 5, 2, 4096),  # 768 pair CTAs: 8 become 128 strips of 128 rows x 32 columns
    (256, [4608], 3, 2, 2184),  # 180 pair CTAs = 152 + 28: 64-column strips over a ragged 136 rows
    (256, [7680], 4, 1, 3000),  # a ragged last row pair (440 rows) in the split-off pairs
    (256, [27648], 4, 1, 768),  # 432 pair CTAs: 128 become 256 x 128 tiles (128 x 128 ones for 128-column pairs)
]


@pytest.mark.parametrize("k,widths,bits,cb,m", SPLIT_CASES, ids=[f"{c[1]}m{c[4]}" for c in SPLIT_CASES])
def test_split_last_wave_byte_equal(k, widths, bits, cb, m):
    """A pair launch with its last wave split off gives the bytes of a single
    launch of one tile shape, and the oracle's values in the split-off region."""
    layer = synthetic.make_layer(k, widths, bits, cb, seed=4400 + m + bits)
    tr, suh, svh = _dev(layer)
    n = layer.n
    x = synthetic.make_x(m, k, seed=4401)
    xh = E.input_transform(x.to(DEV), suh)
    single = B.test_gemm_shape(3, xh, tr, bits, cb, svh, layer.shard_cols)  # 128 x 128 tiles, one launch
    assert single is not None
    for shape in (6, 7, None):  # both pair shapes, and the library's own choice
        got = (E.gemm(xh, tr, bits, cb, svh, layer.shard_cols) if shape is None
               else B.test_gemm_shape(shape, xh, tr, bits, cb, svh, layer.shard_cols))
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), single.view(torch.int16)), f"shape {shape}: bytes differ"
    # the split-off region is the last columns of the last 512 rows
    blocks = [0, n // 128 // 2, n // 128 - 1]
    rows = np.r_[0:8, m - 8:m]
    ref = _oracle(x[rows], layer, blocks)
    got = _np(single)[rows].reshape(len(rows), n // 128, 128)[:, blocks].reshape(len(rows), -1)
    _assert_columns(got, ref)


def test_max_batch_rows():
    """The largest batch the library accepts (2^22 rows): sampled rows against
    the oracle, and rows byte-equal to a small batch of the same inputs."""
    m, k, bits, cb = 1 << 22, 128, 3, 1
    layer = synthetic.make_layer(k, [256], bits, cb, seed=2200)
    x = synthetic.make_x(m, k, seed=2201)
    tr, suh, svh = _dev(layer)
    y = E.gemm(E.input_transform(x.to(DEV), suh), tr, bits, cb, svh, layer.shard_cols)
    torch.cuda.synchronize()
    rows = np.r_[0:16, (m // 2):(m // 2 + 16), (m - 16):m]
    ref = _oracle(x[rows], layer)
    _assert_columns(_np(y)[rows], ref, "max rows")
    small = E.gemm(E.input_transform(x[:300].to(DEV), suh), tr, bits, cb, svh, layer.shard_cols)
    assert torch.equal(small.view(torch.int16), y[:300].view(torch.int16))
    tail = E.gemm(E.input_transform(x[m - 40:].to(DEV), suh), tr, bits, cb, svh, layer.shard_cols)
    assert torch.equal(tail.view(torch.int16), y[m - 40:].view(torch.int16))


@pytest.mark.parametrize("k,widths,bits,cb,split", [
    (1024, [12288], 6, 1, False),  # 96-column strips alone, pairs in the batch
    (512, [384, 384], 4, 2, False),
    (2048, [512], 3, 0, True),
])
def test_each_row_alone_equals_its_row_in_a_batch(k, widths, bits, cb, split):
    """Rows never mix: any row computed on its own has the bytes it has inside a
    300-row batch (not only the batch's first rows)."""
    layer = synthetic.make_layer(k, widths, bits, cb, seed=2300 + k + bits)
    x = synthetic.make_x(300, k, seed=2301)
    y, _ = _run(layer, x, torch.bfloat16, split)
    for r in (0, 17, 150, 299):
        yr, _ = _run(layer, x[r:r + 1], torch.bfloat16, split)
        assert torch.equal(yr.view(torch.int16), y[r:r + 1].view(torch.int16)), f"row {r} differs alone"
