"""Pins of the FP64 oracle to facts other than itself (CPU only).

Each test checks the oracle against something the pages or the mathematics
fix: hand-worked values (tests/golden), closed forms, invariants, an exact
rational model of fp16 rounding, a second bit-serial unpacker, and a naive
loop implementation on tiny shapes.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import exl3_oracle as o
from exl3_trellis_quantized_gb300 import synthetic

CB_ID = {"3inst": 0, "mcg": 1, "mul1": 2}


def _lines(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# ---------------------------------------------------------------------------
# fp16 rounding model (independent: exact rationals)
# ---------------------------------------------------------------------------


def rne_half(fr: Fraction) -> Fraction:
    """Round a rational to binary16, nearest-even (finite range only)."""
    if fr == 0:
        return Fraction(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -14)
    ulp = Fraction(2) ** (e - 10)
    q = a / ulp
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * ulp


def test_half_rounding_matches_exact_model():
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.standard_normal(2000) * 4, rng.standard_normal(500) * 1e-5])
    # exact ties between neighbouring fp16 numbers
    base = o.half_bits_to_f64(rng.integers(0x0400, 0x7800, 300).astype(np.uint16))
    ties = base * (1 + 2.0 ** -11)
    for v in np.concatenate([vals, ties, -ties]):
        got = o.half_bits_to_f64(o.f64_to_half_bits(v))
        assert Fraction(float(got)) == rne_half(Fraction(float(v))), v


# ---------------------------------------------------------------------------
# Codebooks
# ---------------------------------------------------------------------------


def test_codebooks_total_and_bounded():
    s = np.arange(65536)
    for cb in range(3):
        v = o.half_bits_to_f64(o.codebook(cb, s))
        assert np.isfinite(v).all()
    # 3inst / mcg are sums of two halves each in +-[1/8, 2)
    for cb in (0, 1):
        v = o.half_bits_to_f64(o.codebook(cb, s))
        assert np.abs(v).max() < 4.0
    # mul1 values lie between the map's images of t = 0 and t = 1020
    v = o.half_bits_to_f64(o.codebook_mul1(s))
    assert v.min() >= o.MUL1_BIAS - 1e-12
    assert v.max() <= 1020 * o.MUL1_SCALE + o.MUL1_BIAS + 1e-3


def test_codebook_hand_worked_values(golden_dir):
    rows = _lines(golden_dir, "codebook_values.txt")
    assert len(rows) >= 7
    for name, state, bits, value in rows:
        got = int(o.codebook(CB_ID[name], [int(state)])[0])
        assert got == int(bits, 16), (name, state, hex(got))
        assert o.half_bits_to_f64([got])[0] == float(value)


def test_mcg_multiplier_is_the_printed_one():
    # cuda-exl3 README, "GLM-5.3-Flash": multiplier 0xCBAC1FED.
    assert o.MCG_MULT == 0xCBAC1FED
    # every half of the masked word of state 1 comes straight from the multiplier
    u = (0xCBAC1FED & 0x8FFF8FFF) ^ 0x30003000
    lo = Fraction(1) + Fraction(u & 0x3FF, 1024)
    lo *= Fraction(2) ** (((u >> 10) & 0x1F) - 15)
    hi_bits = u >> 16
    hi = Fraction(1) + Fraction(hi_bits & 0x3FF, 1024)
    hi *= Fraction(2) ** (((hi_bits >> 10) & 0x1F) - 15)
    hi *= -1 if hi_bits & 0x8000 else 1
    assert Fraction(float(o.half_bits_to_f64(o.codebook_mcg([1]))[0])) == rne_half(lo + hi)


def test_mul1_single_rounding_exhaustive():
    """All 1021 byte sums: one rounding of t*scale + bias, checked in exact rationals."""
    scale = Fraction(o.MUL1_SCALE)
    bias = Fraction(o.MUL1_BIAS)
    assert scale == rne_half(Fraction(1) / Fraction(1478, 10))
    assert bias == rne_half(Fraction(-510) / Fraction(1478, 10))
    # find a state for every reachable byte sum and compare
    s = np.arange(65536, dtype=np.uint64)
    u = (s * o.MUL1_MULT) & 0xFFFFFFFF
    t = (u & 0xFF) + ((u >> 8) & 0xFF) + ((u >> 16) & 0xFF) + ((u >> 24) & 0xFF)
    vals = o.half_bits_to_f64(o.codebook_mul1(s))
    seen = {}
    for ti, vi in zip(t.tolist(), vals.tolist()):
        seen.setdefault(ti, vi)
    assert len(seen) > 500
    for ti, vi in seen.items():
        assert Fraction(vi) == rne_half(ti * scale + bias), ti


# ---------------------------------------------------------------------------
# Tile layout and unpack
# ---------------------------------------------------------------------------


def test_tile_order_golden(golden_dir):
    for row in _lines(golden_dir, "tile_order.txt"):
        lane = int(row[0])
        for j, kn in enumerate(row[1:]):
            k, n = (int(a) for a in kn.split(","))
            assert o.tile_position(8 * lane + j) == (k, n), (lane, j)


def test_tile_order_is_a_bijection():
    pos = {o.tile_position(v) for v in range(256)}
    assert pos == {(k, n) for k in range(16) for n in range(16)}


def _tile_with_bit(bits, p):
    words = np.zeros(16 * bits, dtype=np.uint16)
    words[p // 16] = 1 << (p % 16)
    return words


def test_single_bit_states_golden(golden_dir):
    for row in _lines(golden_dir, "single_bit_states.txt"):
        bits, p = int(row[0]), int(row[1])
        want = np.zeros(256, dtype=np.uint32)
        for item in row[2:]:
            v, st = item.split(":")
            want[int(v)] = int(st)
        words = _tile_with_bit(bits, p)
        assert np.array_equal(o.trellis_states(words, bits), want), (bits, p)
        assert o.trellis_states_bitserial(words, bits) == want.tolist()


@pytest.mark.parametrize("bits", range(1, 9))
def test_two_unpackers_agree(bits):
    words = synthetic.random_words(16 * bits * 6, seed=100 + bits).numpy().astype(np.uint16)
    tiles = words.reshape(6, 16 * bits)
    fast = o.trellis_states(tiles, bits)
    for i in range(6):
        assert fast[i].tolist() == o.trellis_states_bitserial(tiles[i], bits)


def test_six_bit_lane_window_is_58_bits():
    """At 6 bits the 8 values of lane l depend exactly on the 58 bits [48l-10, 48l+48)."""
    bits = 6
    base = synthetic.random_words(96, seed=7).numpy().astype(np.uint16)
    ref = o.trellis_states(base, bits)
    for lane in (0, 1, 13, 31):
        lo = 48 * lane - 10
        inside = {(lo + i) % 1536 for i in range(58)}
        for p in range(1536):
            w = base.copy()
            w[p // 16] ^= np.uint16(1 << (p % 16))
            changed = not np.array_equal(o.trellis_states(w, bits)[8 * lane:8 * lane + 8],
                                         ref[8 * lane:8 * lane + 8])
            assert changed == (p in inside), (lane, p)


def test_dequantize_places_tiles():
    """Tile (kt, nt) lands at rows 16kt.., columns 16nt.. with the fragment order."""
    bits, cb = 3, 1
    tr = synthetic.random_trellis(32, 48, bits, __import__("torch").Generator().manual_seed(3)).numpy()
    w = o.dequantize(tr, bits, cb)
    assert w.shape == (32, 48)
    for kt in range(2):
        for nt in range(3):
            st = o.trellis_states_bitserial(tr[kt, nt], bits)
            vals = o.half_bits_to_f64(o.codebook(cb, st))
            for v in (0, 1, 2, 7, 8, 100, 255):
                k, n = o.tile_position(v)
                assert w[16 * kt + k, 16 * nt + n] == vals[v]


# ---------------------------------------------------------------------------
# Hadamard, scales and the full layer
# ---------------------------------------------------------------------------


def test_hadamard_orthogonal_and_symmetric():
    h = o.hadamard128()
    assert np.array_equal(h @ h, 128 * np.eye(128))
    assert np.array_equal(h, h.T)
    assert h[0].sum() == 128 and h[:, 0].sum() == 128
    # Sylvester recursion H_2n = [[H, H], [H, -H]]
    assert np.array_equal(h[:64, 64:], h[:64, :64]) and np.array_equal(h[64:, 64:], -h[:64, :64])


def test_input_transform_unit_vectors_and_double_application():
    k = 256
    x = np.zeros((1, k))
    x[0, 130] = 1.0
    xh = o.input_transform(x, np.ones(k))[0, 0]
    h = o.hadamard128()
    assert np.array_equal(xh[128:], h[:, 2] / 16) and not xh[:128].any()
    # applying the rotation twice gives x * 128 * 2^-8 = x / 2
    r = np.random.default_rng(3).standard_normal((3, k))
    twice = o.input_transform(o.input_transform(r, np.ones(k))[0], np.ones(k))[0]
    assert np.allclose(twice, r / 2, rtol=0, atol=1e-12)


def test_scales_make_identity_weights_orthonormal():
    """2^-4 * 2^-3 * 128 = 1: with Wq = I the layer is y = x * suh * svh."""
    k = 256
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5, k))
    suh = rng.uniform(0.8, 1.2, k) * rng.choice([-1, 1], k)
    svh = rng.uniform(0.8, 1.2, k) * rng.choice([-1, 1], k)
    y = o.linear_dense(x, np.eye(k), suh, svh, [0, k])
    assert np.allclose(y, x * suh * svh, rtol=1e-13, atol=1e-13)


def test_permutation_weights_catch_transposition():
    """Wq[k, n] = 1 iff n = pi(k): y = svh * H(H(x*suh)/16 permuted)/8."""
    k = 128
    rng = np.random.default_rng(5)
    pi = rng.permutation(k)
    w = np.zeros((k, k))
    w[np.arange(k), pi] = 1.0
    x = rng.standard_normal((2, k))
    h = o.hadamard128()
    xh = (x @ h.T) / 16
    z = np.zeros_like(xh)
    z[:, pi] = xh
    want = (z @ h.T) / 8
    assert np.allclose(o.linear_dense(x, w, np.ones(k), np.ones(k), [0, k]), want, atol=1e-12)
    assert not np.allclose(o.linear_dense(x, w.T, np.ones(k), np.ones(k), [0, k]), want, atol=1e-3)


@pytest.mark.parametrize("cb", [0, 1, 2])
def test_constant_trellis_closed_form(cb):
    """All-zero words give state 0 everywhere, so Wq = c * ones and
    y[r, n] = svh[n] * 2^-3 * 128 * c * 2^-4 * 128 * sum_b (x*suh)[r, 128b] for n % 128 == 0, else 0."""
    k, n, bits = 256, 256, 4
    tr = np.zeros((k // 16, n // 16, 16 * bits), dtype=np.int16)
    c = o.half_bits_to_f64(o.codebook(cb, [0]))[0]
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, k))
    suh = rng.uniform(0.8, 1.2, (1, k))
    svh = rng.uniform(0.8, 1.2, n)
    y = o.linear(x, tr, bits, cb, suh, svh, [0, n])
    xs = x * suh[0]
    s = xs[:, 0] + xs[:, 128]
    want = np.zeros((3, n))
    for blk in range(n // 128):
        want[:, 128 * blk] = svh[128 * blk] * 2.0 ** -3 * 128 * c * 2.0 ** -4 * 128 * s
    assert np.allclose(y, want, rtol=1e-12, atol=1e-9)


@pytest.mark.parametrize("bits", range(1, 9))
@pytest.mark.parametrize("cb", [0, 1, 2])
def test_linear_matches_bruteforce(bits, cb):
    kk, nn = (128, 256) if bits % 2 else (256, 128)
    layer = synthetic.make_layer(kk, [nn], bits, cb, seed=200 + 10 * bits + cb)
    x = synthetic.make_x(2, kk, seed=300 + bits).float().numpy()
    args = (layer.trellis.numpy(), bits, cb, layer.suh.float().numpy(), layer.svh.float().numpy(), layer.shard_cols)
    fast = o.linear(x, *args)
    slow = o.linear_bruteforce(x, *args)
    assert np.allclose(fast, slow, rtol=1e-12, atol=1e-12 * np.abs(slow).max())


def test_fused_shards_equal_separate_layers():
    """A fused launch equals each shard computed alone on its column slice."""
    k, bits, cb = 256, 5, 2
    layer = synthetic.make_layer(k, [128, 256], bits, cb, seed=9)
    x = synthetic.make_x(3, k, seed=9).float().numpy()
    tr = layer.trellis.numpy()
    suh = layer.suh.float().numpy()
    svh = layer.svh.float().numpy()
    fused = o.linear(x, tr, bits, cb, suh, svh, layer.shard_cols)
    a = o.linear(x, tr[:, :8], bits, cb, suh[0:1], svh[:128], [0, 128])
    b = o.linear(x, tr[:, 8:], bits, cb, suh[1:2], svh[128:], [0, 256])
    assert np.array_equal(fused, np.concatenate([a, b], axis=1))


def test_column_block_selection_matches_full():
    layer = synthetic.make_layer(128, [384], 2, 0, seed=11)
    x = synthetic.make_x(2, 128, seed=11).float().numpy()
    args = (layer.trellis.numpy(), 2, 0, layer.suh.float().numpy(), layer.svh.float().numpy(), layer.shard_cols)
    full = o.linear(x, *args)
    part = o.linear(x, *args, col_blocks=[2, 0])
    assert np.array_equal(part, np.concatenate([full[:, 256:], full[:, :128]], axis=1))


# ---------------------------------------------------------------------------
# SwiGLU folded into the down-projection's input transform
# ---------------------------------------------------------------------------


def test_swiglu_closed_forms():
    g = np.array([[0.0, 1.0, -1.0, 3.0, -40.0, 40.0, -800.0]])
    up = np.array([[2.0, 1.0, 1.0, -0.5, 1.0, 1.0, 1.0]])
    h = o.swiglu(np.concatenate([g, up], axis=1))
    assert h[0, 0] == 0.0  # silu(0) = 0
    assert h[0, 1] == pytest.approx(1.0 / (1.0 + np.exp(-1.0)), rel=1e-15)  # sigmoid(1)
    assert h[0, 2] == pytest.approx(-1.0 / (1.0 + np.e), rel=1e-15)  # -sigmoid(-1)
    assert h[0, 3] == pytest.approx(-0.5 * 3.0 / (1.0 + np.exp(-3.0)), rel=1e-15)  # times up
    assert abs(h[0, 4]) < 1e-15 and h[0, 5] == pytest.approx(40.0, rel=1e-15)  # tails: 0 and identity
    assert h[0, 6] == 0.0  # e^800 overflows: the result is a signed zero, not a NaN


def test_swiglu_identities():
    """silu(g) - silu(-g) = g (sigmoid(g) + sigmoid(-g) = 1), and silu agrees with
    the independent form g/2 * (1 + tanh(g/2)); a dropped factor, a sign error
    in the exponent or swapped gate/up halves fails one of these."""
    g = np.linspace(-12.0, 12.0, 2001)[None]
    one = np.ones_like(g)
    pos = o.swiglu(np.concatenate([g, one], axis=1))
    neg = o.swiglu(np.concatenate([-g, one], axis=1))
    assert np.allclose(pos - neg, g, rtol=0, atol=1e-12)
    assert np.allclose(pos, g / 2 * (1 + np.tanh(g / 2)), rtol=1e-13, atol=1e-15)
    # gate and up are not interchangeable: the gate goes through silu, up does not
    up = np.full_like(g, 3.0)
    assert np.allclose(o.swiglu(np.concatenate([g, up], axis=1)), 3.0 * pos, rtol=1e-15, atol=0)


def test_swiglu_transform_is_the_transform_of_swiglu():
    gu = synthetic.make_x(9, 512, seed=61).double().numpy()
    suh = np.random.default_rng(62).uniform(0.5, 1.5, (2, 256))
    assert np.array_equal(o.input_transform_swiglu(gu, suh), o.input_transform(o.swiglu(gu), suh))


# ---------------------------------------------------------------------------
# Mixture of experts: grouped rows through each block's expert
# ---------------------------------------------------------------------------


def _moe_case(seed=71, tokens=7, experts=5, topk=2, block=4):
    layer = synthetic.make_moe_layer(256, [128, 128], 3, 1, experts, seed=seed)
    routing = synthetic.make_routing(tokens, experts, topk, block, seed=seed + 1)
    x = synthetic.make_x(tokens, 256, seed=seed + 2).double().numpy()
    return layer, routing, x


def test_routing_holds_every_pair_once():
    _, r, _ = _moe_case()
    ids = r.sorted_ids.numpy()
    live = ids[ids < r.num_tokens * r.topk]
    assert sorted(live.tolist()) == list(range(r.num_tokens * r.topk))
    assert r.rows % r.block == 0 and len(r.block_expert) == r.rows // r.block
    assert (r.block_expert.numpy() == -1).sum() == 2


def test_moe_rows_follow_topk_choices():
    """Row of pair (t, j) equals the dense layer of expert topk_ids[t, j] on token
    t, found through the routing's own top-k table rather than the block ids."""
    layer, r, x = _moe_case()
    y = o.moe_linear(x, r.sorted_ids.numpy(), r.block_expert.numpy(), r.block, r.topk, layer.trellis.numpy(),
                     layer.bits, layer.codebook, layer.suh.double().numpy(), layer.svh.double().numpy(),
                     layer.shard_cols)
    ids = r.sorted_ids.numpy()
    for row, pair in enumerate(ids):
        if pair >= r.num_tokens * r.topk:
            continue
        t, j = divmod(int(pair), r.topk)
        e = int(r.topk_ids[t, j])
        want = o.linear(x[t][None], layer.trellis[e].numpy(), layer.bits, layer.codebook,
                        layer.suh[e].double().numpy(), layer.svh[e].double().numpy(), layer.shard_cols)[0]
        assert np.allclose(y[row], want, rtol=0, atol=1e-12)
    blocks = r.block_expert.numpy()
    for b, e in enumerate(blocks):
        rows = y[b * r.block:(b + 1) * r.block]
        if e < 0:
            assert np.isnan(rows).all()  # skipped: never written
        else:
            pad = ids[b * r.block:(b + 1) * r.block] >= r.num_tokens * r.topk
            assert (rows[pad] == 0).all()


def test_moe_input_transform_follows_topk_choices():
    layer, r, x = _moe_case()
    xh = o.moe_input_transform(x, r.sorted_ids.numpy(), r.block_expert.numpy(), r.block, r.topk,
                               layer.suh.double().numpy())
    ids = r.sorted_ids.numpy()
    for row, pair in enumerate(ids):
        if pair >= r.num_tokens * r.topk:
            assert (xh[:, row] == 0).all()
            continue
        t, j = divmod(int(pair), r.topk)
        e = int(r.topk_ids[t, j])
        assert np.array_equal(xh[:, row], o.input_transform(x[t][None], layer.suh[e].double().numpy())[:, 0])


# ---------------------------------------------------------------------------
# Mixture of experts: the weighted combine of a token's top-k rows
# ---------------------------------------------------------------------------


def _moe_rows(layer, r, x):
    return o.moe_linear(x, r.sorted_ids.numpy(), r.block_expert.numpy(), r.block, r.topk, layer.trellis.numpy(),
                        layer.bits, layer.codebook, layer.suh.double().numpy(), layer.svh.double().numpy(),
                        layer.shard_cols)


def _combine(y, r, w, experts, block_expert=None):
    be = r.block_expert.numpy() if block_expert is None else block_expert
    return o.moe_combine(y, r.sorted_ids.numpy(), be, r.block, r.topk, w, r.num_tokens, experts)


def test_moe_combine_is_the_weighted_sum_of_dense_experts():
    """out[t] = sum_j w[t, j] * layer_{topk_ids[t, j]}(x[t]), with the experts taken
    from the routing's own top-k table, not from the block layout (the rows of
    blocks of no expert are NaN in the grouped output: reading one would show)."""
    layer, r, x = _moe_case()
    w = synthetic.make_topk_weights(r.num_tokens, r.topk, seed=81).double().numpy()
    out = _combine(_moe_rows(layer, r, x), r, w, 5)
    for t in range(r.num_tokens):
        want = np.zeros(out.shape[1])
        for j in range(r.topk):
            e = int(r.topk_ids[t, j])
            want += w[t, j] * o.linear(x[t][None], layer.trellis[e].numpy(), layer.bits, layer.codebook,
                                       layer.suh[e].double().numpy(), layer.svh[e].double().numpy(),
                                       layer.shard_cols)[0]
        assert np.allclose(out[t], want, rtol=0, atol=1e-12)


def test_moe_combine_one_hot_weights_gather_the_slot_row():
    layer, r, x = _moe_case(seed=91, tokens=6, experts=4, topk=3, block=4)
    y = _moe_rows(layer, r, x)
    ids = r.sorted_ids.numpy()
    for j in range(r.topk):
        w = np.zeros((r.num_tokens, r.topk))
        w[:, j] = 1.0
        out = _combine(y, r, w, 4)
        for t in range(r.num_tokens):
            (row,) = np.nonzero(ids == t * r.topk + j)[0]
            assert np.array_equal(out[t], y[row])


def test_moe_combine_ignores_the_block_layout():
    """The same choices with or without blocks of no expert between the live
    ones give the same combine."""
    layer = synthetic.make_moe_layer(256, [128, 128], 3, 1, 5, seed=101)
    x = synthetic.make_x(7, 256, seed=102).double().numpy()
    w = synthetic.make_topk_weights(7, 2, seed=103).double().numpy()
    outs = []
    for empty in (0, 3):
        r = synthetic.make_routing(7, 5, 2, 4, seed=104, empty_blocks=empty)
        outs.append(_combine(_moe_rows(layer, r, x), r, w, 5))
    assert np.array_equal(outs[0], outs[1])


def test_moe_combine_drops_pairs_without_a_live_row():
    """Marking a live block as no expert (-1, or an id past the last expert)
    removes exactly its pairs' terms."""
    layer, r, x = _moe_case(seed=111)
    w = synthetic.make_topk_weights(r.num_tokens, r.topk, seed=112).double().numpy()
    y = _moe_rows(layer, r, x)
    full = _combine(y, r, w, 5)
    be = r.block_expert.numpy().copy()
    b = int(np.nonzero(be >= 0)[0][0])
    for mark in (-1, 5):
        dropped = be.copy()
        dropped[b] = mark
        got = _combine(y, r, w, 5, dropped)
        want = full.copy()
        for row in range(b * r.block, (b + 1) * r.block):
            pair = int(r.sorted_ids[row])
            if pair < r.num_tokens * r.topk:
                t, j = divmod(pair, r.topk)
                want[t] -= w[t, j] * y[row]
        assert np.allclose(got, want, rtol=0, atol=1e-12)
