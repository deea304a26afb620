"""The cost model's tile plan (host only, no GPU): pins of the decisions the
GEMM's measured shape costs lead to on a 152-SM GB300, and the invariants of a
split last wave (the first launch is whole waves; the second covers exactly the
pair tiles left)."""
import pytest

from exl3_trellis_quantized_gb300 import binding as B

SMS = 152  # the plan uses the current device's SM count, 152 without one
(N32S, N64S, N128S, N128, N128R2, N256R2, N128R2P, N256R2P, N128SK4, N96SK4, N96, N96R2, N32SK8, N64SK4, N96M64K4,
 N64M64K4, N64K4, N32K4, T128K4, T128, S96K4, T128K4X16, S96K4X16, T128X16, T128K4X64, T128X64, T128X128, S96K4X64,
 T128K4X128) = range(29)
PAIR_BN = {N128R2P: 128, N256R2P: 256}


def plan(m, k, n, cols=None, split=False):
    return B.test_tile_plan(m, k, n, cols or [0, n], split)


@pytest.mark.parametrize("m,want", [
    # 96 column blocks: 96-column strips on 128 SMs, the decoded weights as
    # the tensor core's 128-row operand, 16-row tiles up to 16 rows
    (1, (S96K4X16, -1, 0, 0, 0)), (16, (S96K4X16, -1, 0, 0, 0)), (32, (S96K4, -1, 0, 0, 0)),
    (48, (S96K4X64, -1, 0, 0, 0)), (64, (S96K4X64, -1, 0, 0, 0)),  # 64-row swapped strips, four atoms a stage
    (128, (N96, -1, 0, 0, 0)), (256, (N96R2, -1, 0, 0, 0)),
    (512, (N256R2P, -1, 0, 0, 0)),  # 96 pair CTAs: one partial wave, nothing to split off
    (1024, (N256R2P, N128R2P, 76, 512, 7168)),  # 192 = 152 + 40 CTAs: the 40 become 40 pairs of 256x128 tiles
    (4096, (N256R2P, N32K4, 380, 3584, 11264)),  # 768 = 5 x 152 + 8: the 8 become 128 strips of 128 x 32
])
def test_q_proj_plan(m, want):
    assert plan(m, 5120, 12288) == want


@pytest.mark.parametrize("m,k,n,cols,want", [
    (64, 12288, 4096, None, N32K4), (100, 12288, 4096, None, N32K4),  # 32 blocks: 128 strips of 32 columns
    (64, 4096, 8192, None, N64M64K4), (100, 4096, 8192, None, N64K4),  # 64 blocks: 64-column strips, four atoms
    (64, 12416, 4096, None, N128), (100, 12416, 4096, None, N128),  # odd k/128: no four-atom strips
    (64, 4096, 2048, None, N32K4),  # 16 blocks: 64 strips of 32 columns
    (128, 5120, 6144, None, N64K4), (100, 5120, 12288, None, N96),
    # wide layers: the tensor-memory kernel holding 64 or 128 rows (four atoms
    # a stage when k/128 is even) where its persistent waves beat 256-column tiles
    (48, 5120, 34816, [0, 17408, 34816], T128K4X64), (64, 4096, 154880, None, T128K4X64),
    (128, 4096, 154880, None, T128K4X128), (100, 4096, 154880, None, T128K4X128),
    (128, 5120, 34816, [0, 17408, 34816], T128K4X128),  # two waves of items, still ahead of 256-column tiles
    (48, 4224, 154880, None, T128X128),  # odd k/128: no four-atom tiles, the 128-row items on two
])
def test_mid_batch_plan(m, k, n, cols, want):
    assert plan(m, k, n, cols)[0] == want


def test_narrow_and_split_layers():
    assert plan(16, 12288, 4096)[0] == N32SK8  # 32 column blocks: 32-column strips on 128 SMs, 8 atoms a stage
    assert plan(16, 2048, 4096)[0] == N32SK8  # k = 2048 holds four stages of eight atoms
    assert plan(32, 2048, 4096)[0] == N32SK8
    # 272 blocks fill the GPU at 128 columns: the persistent tensor-memory kernel
    assert plan(16, 5120, 34816, [0, 17408, 34816])[0] == T128K4X16
    assert plan(32, 5120, 34816, [0, 17408, 34816])[0] == T128K4
    assert plan(16, 4096, 154880)[0] == T128K4X16
    assert plan(16, 4224, 154880)[0] == T128X16  # odd k/128: two atoms a stage
    assert plan(16, 4096, 8192)[0] == N64SK4  # 64 blocks: 64-column strips, four atoms a stage
    assert plan(16, 384, 4096)[0] != N32S  # odd k/128: no four-atom tiles
    # split-k at m <= 32: the tensor-memory kernel over (block, part) items,
    # four atoms a stage when the parts are whole 256-row units of k (k/128
    # even and P <= k/256), else two
    assert plan(1, 17408, 5120, split=True)[0] == T128K4X16  # 7 parts of 68 units
    assert plan(32, 12288, 4096, split=True)[0] == T128K4  # 9 parts of 48 units
    assert plan(16, 1024, 512, split=True)[0] == T128X16  # 8 parts > 4 units
    assert plan(32, 2048, 4096, split=True)[0] == T128  # 9 parts > 8 units
    # 33-128 rows: there too when a CTA's items hold >= 1024 k in all
    assert plan(64, 17408, 5120, split=True)[0] == T128K4X64  # 2 waves of 2487-deep parts
    assert plan(128, 5120, 6144, split=True)[0] == T128K4X128  # 1 wave of 1707-deep parts
    assert plan(64, 2048, 4096, split=True)[0] == N256R2  # 2 x 228 k: shared-memory tiles
    assert plan(128, 4096, 1024, split=True)[0] == N128  # 1 x 256 k


@pytest.mark.parametrize("m,k,n", [(1024, 5120, 12288), (4096, 5120, 12288), (2048, 5120, 34816),
                                   (4096, 5120, 34816), (3000, 4096, 7680), (1500, 2048, 20480)])
def test_split_last_wave_invariants(m, k, n):
    shape, tail, primary, row_base, col_base = plan(m, k, n)
    if shape not in PAIR_BN or tail < 0:
        return
    bn = PAIR_BN[shape]
    rows_per_pair_tile = 512
    ncol = n // bn
    nrp = -(-m // rows_per_pair_tile)
    total_tiles = ncol * nrp
    assert (2 * primary) % SMS == 0, "the first launch is whole waves"
    assert row_base == (nrp - 1) * rows_per_pair_tile, "the split-off tiles are in the last row pair"
    assert (n - col_base) // bn == total_tiles - primary, "the second launch covers exactly the tiles left"
    assert col_base % bn == 0 and tail in (N128, N128R2, N256R2, N128R2P, N64K4, N32K4)


def test_plan_rejects_invalid():
    with pytest.raises(B.Exl3Error):
        B.test_tile_plan(0, 5120, 12288, [0, 12288])
    with pytest.raises(B.Exl3Error):
        B.test_tile_plan(16, 5000, 12288, [0, 12288])
    with pytest.raises(B.Exl3Error):
        B.test_tile_plan(16, 5120, 12288, [0, 100, 12288])


TAIL_BN = {N128: 128, N128R2: 128, N256R2: 256, N128R2P: 128, N64K4: 64, N32K4: 32}


@pytest.mark.parametrize("k", [2048, 2176, 5120], ids=["k2048", "k2176_odd_blocks", "k5120"])
@pytest.mark.parametrize("split_shards", [False, True], ids=["one_shard", "two_shards"])
def test_split_plans_hold_over_a_grid(k, split_shards):
    """Every split plan over a grid of widths and batch sizes: the first launch
    is whole waves, the second covers exactly the pair tiles left, its tiles
    divide the split-off columns and every shard edge, and four-atom strips only
    appear when k holds an even number of 128-row blocks."""
    checked = 0
    for n in range(2048, 40961, 1024):
        cols = [0, n // 2 // 128 * 128, n] if split_shards else [0, n]
        for m in range(520, 8193, 184):
            shape, tail, primary, row_base, col_base = plan(m, k, n, cols)
            if tail < 0:
                continue
            bn = PAIR_BN[shape]
            ncol, nrp = n // bn, -(-m // 512)
            assert (2 * primary) % SMS == 0
            assert row_base == (nrp - 1) * 512
            assert (n - col_base) // bn == ncol * nrp - primary
            tb = TAIL_BN[tail]
            assert (n - col_base) % tb == 0 and col_base % 128 == 0
            assert all(c % max(tb, 128) == 0 for c in cols), (n, m, tail, cols)
            if tail in (N64K4, N32K4):
                assert (k // 128) % 2 == 0
            checked += 1
    assert checked > 20
