"""Plain FP64 CPU oracle of the EXL3 trellis-quantized linear layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
link this module: only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA
implementation; both sides only consume the seeded inputs of
``exl3_trellis_quantized_gb300.synthetic``.

What it computes (the layer's plain definition)::

    x'_s[r, :] = H_K(x[r, :] * suh_s) * 2^-4           (input rotation)
    z[r, n]    = sum_k x'_{s(n)}[r, k] * Wq[k, n]         (contraction)
    y[r, :]    = (H_N(z[r, :]) * 2^-3) * svh               (output rotation)

with H_K / H_N the block-diagonal 128-point Sylvester Hadamard matrix and
Wq the weights decoded from 16x16 trellis tiles.  Sources: TensorFold PR #740
("Arithmetic", steps 1-3); cuda-exl3 README ("Why custom kernels",
"One op per layer", "Notes on the format", "Tensor parallel", "Loading into a
dim vLLM has padded").  Everything is done in float64: the rotated input is
not rounded to fp16 and the output is not rounded to bf16/fp16, so the
oracle is the exact result up to float64 rounding.

The pages fix the tile shape, the bit widths, the codebook names, the mcg
multiplier and the rounding rules, but not the bit order of the trellis
stream, the position of a state's window, nor the 3inst/mul1 constants.
Where they are silent this module takes one plain reading, stated at each
function.  These readings are pinned against closed forms, hand-worked
values and a second, bit-serial unpacker in ``tests/test_oracle_pins.py``;
parity with real EXL3 checkpoints is unpinned (no checkpoint or printed
codebook value exists to check against).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

# ---------------------------------------------------------------------------
# fp16 helpers
# ---------------------------------------------------------------------------


def half_bits_to_f64(bits) -> np.ndarray:
    """Value of IEEE binary16 bit patterns, exactly, as float64."""
    b = np.asarray(bits, dtype=np.uint16)
    return b.view(np.float16).astype(np.float64)


def f64_to_half_bits(x) -> np.ndarray:
    """Round float64 values to binary16, nearest-even, once; return bits."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


# ---------------------------------------------------------------------------
# Codebooks: 16-bit trellis state -> one fp16 weight
# ---------------------------------------------------------------------------

# mcg multiplier, printed with the GLM-5.3-Flash checkpoint description
# (cuda-exl3 README, section "GLM-5.3-Flash").
MCG_MULT = 0xCBAC1FED

# Reading (the pages give no 3inst or mul1 constants): 3inst is the mcg map
# with an increment, i.e. one multiply-add, the mask/xor and the half add
# (which is what the codebook's name suggests); mul1 uses the same multiplier.
INST3_MULT = 0xCBAC1FED
INST3_ADD = 1
MUL1_MULT = 0xCBAC1FED

# Reading: the mask keeps sign, the two low exponent bits and the mantissa of
# each 16-bit half; the xor sets the exponent field to 0b011xx, so each half
# lies in +-[2^-3, 2).  This makes every state decode to a finite value, the
# totality the cuda-exl3 README states for all 65,536 states of every codebook
# ("Loading into a dim vLLM has padded").
HALF_MASK = 0x8FFF8FFF
HALF_XOR = 0x30003000

# Reading for mul1 (TensorFold PR, "Arithmetic": the value comes from one fp16
# fused multiply-add applied to an exactly computed sum, so it is rounded once):
# the exact sum is the sum of the four bytes of the hashed state (0..1020);
# the affine map standardises a sum of four uniform bytes (mean 510,
# sd sqrt(4*(256^2-1)/12) ~= 147.8).  Both coefficients are fp16 numbers.
MUL1_SCALE = float(np.float16(1.0 / 147.8))
MUL1_BIAS = float(np.float16(-510.0 / 147.8))


def _as_states(states) -> np.ndarray:
    s = np.asarray(states, dtype=np.uint64)
    if np.any(s >= (1 << 16)):
        raise ValueError("trellis states are 16-bit")
    return s


def _sum_of_halves(u: np.ndarray) -> np.ndarray:
    """fp16 value of half(u & 0xffff) + half(u >> 16), rounded once."""
    u = (u & HALF_MASK) ^ HALF_XOR
    lo = half_bits_to_f64((u & 0xFFFF).astype(np.uint16))
    hi = half_bits_to_f64((u >> 16).astype(np.uint16))
    # Two binary16 numbers add exactly in float64; round the sum to fp16 once.
    return f64_to_half_bits(lo + hi)


def codebook_3inst(states) -> np.ndarray:
    """3inst: u = (a*s + c) mod 2^32, masked to two halves, halves summed."""
    s = _as_states(states)
    u = (s * INST3_MULT + INST3_ADD) & 0xFFFFFFFF
    return _sum_of_halves(u)


def codebook_mcg(states) -> np.ndarray:
    """mcg: u = (0xCBAC1FED * s) mod 2^32, masked to two halves, halves summed."""
    s = _as_states(states)
    u = (s * MCG_MULT) & 0xFFFFFFFF
    return _sum_of_halves(u)


def codebook_mul1(states) -> np.ndarray:
    """mul1: t = byte sum of (m * s) mod 2^32; value = fp16(t*scale + bias), one rounding."""
    s = _as_states(states)
    u = (s * MUL1_MULT) & 0xFFFFFFFF
    t = (u & 0xFF) + ((u >> 8) & 0xFF) + ((u >> 16) & 0xFF) + ((u >> 24) & 0xFF)
    # t*scale + bias is exact in float64 (t < 2^10, both coefficients fp16);
    # the single rounding is the cast to fp16.
    return f64_to_half_bits(t.astype(np.float64) * MUL1_SCALE + MUL1_BIAS)


CODEBOOKS = {0: codebook_3inst, 1: codebook_mcg, 2: codebook_mul1}
CODEBOOK_NAMES = {0: "3inst", 1: "mcg", 2: "mul1"}


def codebook(cb: int, states) -> np.ndarray:
    return CODEBOOKS[int(cb)](states)


# ---------------------------------------------------------------------------
# Tile layout and trellis unpack
# ---------------------------------------------------------------------------


def tile_position(v: int):
    """(k, n) inside a 16x16 tile of the tile's v-th decoded value.

    Tiles decode directly into the B operands of two mma.m16n8k16
    instructions, which fixes the value order (TensorFold PR, "Arithmetic"
    step 2), each lane holding 8 consecutive values (cuda-exl3 README, "Where the time
    goes": lane*8 alignment).  Lane l = v // 8 holds, for each n8 half h,
    the fragment registers b0 = (k = 2q, 2q+1) and b1 = (k = 2q+8, 2q+9) of
    column n = l // 4 + 8h, with q = l % 4.  Reading: the 8 values of a lane
    are ordered h-major, then register, then element.
    """
    lane, w = divmod(int(v), 8)
    h, e = divmod(w, 4)
    g, q = divmod(lane, 4)
    k = 2 * q + (e & 1) + 8 * (e >> 1)
    n = g + 8 * h
    return k, n


TILE_K = np.zeros(256, dtype=np.int64)
TILE_N = np.zeros(256, dtype=np.int64)
for _v in range(256):
    TILE_K[_v], TILE_N[_v] = tile_position(_v)


def _stream_bits(words: np.ndarray) -> np.ndarray:
    """Bits of each tile's word stream, position p = 16*word + bit (LSB first).

    Reading: the tile's 16*bits int16 words form one little-endian bit
    stream; bit p is bit (p mod 16) of word p // 16.
    """
    w = np.ascontiguousarray(words.astype(np.uint16))
    as_bytes = w.view(np.uint8).reshape(*w.shape[:-1], w.shape[-1] * 2)
    if as_bytes.dtype.byteorder == ">":  # pragma: no cover - big-endian hosts only
        raise RuntimeError("little-endian host expected")
    return np.unpackbits(as_bytes, axis=-1, bitorder="little")


def trellis_states(words, bits: int) -> np.ndarray:
    """16-bit state of every value of every tile: ``[..., 16*bits] -> [..., 256]``.

    Reading of the bitshift trellis (cuda-exl3 README, "Where the time
    goes": a lane's 8 values at 6 bits need a 58-bit window = 7*6 + 16, and
    the index math wraps modulo the 48 words of a 6-bit tile): state v is the
    16 bits that end just before position (v+1)*bits of the tile's circular
    stream of 256*bits bits, least significant bit first::

        state_v = sum_{t=0}^{15} bit(((v+1)*bits - 16 + t) mod 256*bits) << t
    """
    if not 1 <= bits <= 8:
        raise ValueError("bits must be 1..8")
    words = np.asarray(words)
    if words.shape[-1] != 16 * bits:
        raise ValueError("last axis must hold 16*bits words")
    stream = _stream_bits(words)  # [..., 256*bits] uint8
    length = 256 * bits
    v = np.arange(256)[:, None]
    t = np.arange(16)[None, :]
    pos = ((v + 1) * bits - 16 + t) % length  # [256, 16]
    gathered = stream[..., pos].astype(np.uint32)  # [..., 256, 16]
    return (gathered << np.arange(16, dtype=np.uint32)).sum(axis=-1, dtype=np.uint32)


def trellis_states_bitserial(tile_words, bits: int) -> list:
    """Second, independent unpacker of ONE tile, as a 16-bit shift register.

    Bits enter at the top (bit 15) and shift toward bit 0.  The register is
    primed with the last 16 bits of the tile's stream (the stream is
    circular), then for each value the next ``bits`` bits are shifted in and
    the register is the value's state.  Pure Python, for small cases only.
    """
    words = [int(w) & 0xFFFF for w in tile_words]
    if len(words) != 16 * bits:
        raise ValueError("a tile holds 16*bits words")
    length = 256 * bits

    def bit(p: int) -> int:
        return (words[p // 16] >> (p % 16)) & 1

    reg = 0
    for p in range(length - 16, length):
        reg = (reg >> 1) | (bit(p) << 15)
    states = []
    p = 0
    for _ in range(256):
        for _ in range(bits):
            reg = (reg >> 1) | (bit(p) << 15)
            p += 1
        states.append(reg)
    return states


def dequantize(trellis, bits: int, cb: int, col_blocks: Optional[Sequence[int]] = None) -> np.ndarray:
    """Wq as float64 [K, N] (or [K, 128*len(col_blocks)] for selected 128-column blocks).

    Tile (kt, nt) of the ``[K/16, N/16, 16*bits]`` trellis covers rows
    16*kt..16*kt+15 and columns 16*nt..16*nt+15 of Wq (TensorFold PR, "What
    it adds"; reading: C order of the printed shape).
    """
    tr = np.asarray(trellis)
    kt, nt, _ = tr.shape
    if col_blocks is not None:
        sel = np.concatenate([np.arange(8 * c, 8 * c + 8) for c in col_blocks])
        tr = tr[:, sel, :]
        nt = tr.shape[1]
    states = trellis_states(tr.astype(np.uint16), bits)  # [kt, nt, 256]
    vals = half_bits_to_f64(codebook(cb, states.reshape(-1)).reshape(states.shape))
    w = np.zeros((kt, 16, nt, 16), dtype=np.float64)
    w[:, TILE_K, :, TILE_N] = np.moveaxis(vals, 2, 0)
    return w.reshape(kt * 16, nt * 16)


# ---------------------------------------------------------------------------
# Hadamard rotations and the full layer
# ---------------------------------------------------------------------------


def hadamard128() -> np.ndarray:
    """Unnormalised 128-point Sylvester Hadamard matrix, H[i, j] = (-1)^popcount(i & j).

    Reading: natural (Sylvester) order, applied to contiguous 128-element
    blocks (cuda-exl3 README, "Tensor parallel" and "Loading into a dim vLLM
    has padded").
    """
    i = np.arange(128)
    pc = np.vectorize(lambda a: bin(int(a)).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1.0, -1.0)


_H128 = hadamard128()


def blockwise_hadamard(v: np.ndarray) -> np.ndarray:
    """Apply H128 to each contiguous 128-block of the last axis (float64)."""
    v = np.asarray(v, dtype=np.float64)
    if v.shape[-1] % 128:
        raise ValueError("length must be a multiple of 128")
    blocks = v.reshape(*v.shape[:-1], v.shape[-1] // 128, 128)
    return (blocks @ _H128.T).reshape(v.shape)


def input_transform(x, suh) -> np.ndarray:
    """x' = H(x * suh) * 2^-4 per shard, float64 [S, m, K] (TensorFold PR, "Arithmetic" step 1)."""
    x = np.asarray(x, dtype=np.float64)
    suh = np.atleast_2d(np.asarray(suh, dtype=np.float64))
    return np.stack([blockwise_hadamard(x * suh[s][None, :]) * 2.0 ** -4 for s in range(suh.shape[0])])


def swiglu(gate_up) -> np.ndarray:
    """h = silu(gate) * up, float64 [m, K] from gate_up [m, 2K].

    The down-projection's input of a gated MLP, folded into its input
    transform (cuda-exl3 README, "MoE throughput": SwiGLU folded into the
    down-projection's input transform).  The pages print no formula; this
    module reads it as the usual SwiGLU, silu(g) * u with silu(g) = g / (1 +
    e^-g), gate in the first K columns and up in the last K (the column order
    of a gate_up layer fused as two shards).
    """
    gu = np.asarray(gate_up, dtype=np.float64)
    k = gu.shape[1] // 2
    g, u = gu[:, :k], gu[:, k:]
    with np.errstate(over="ignore"):  # e^-g overflows to inf for very negative g: silu -> -0
        return g / (1.0 + np.exp(-g)) * u


def input_transform_swiglu(gate_up, suh) -> np.ndarray:
    """x' = H(swiglu(gate_up) * suh) * 2^-4 per shard, float64 [S, m, K]."""
    return input_transform(swiglu(gate_up), suh)


def output_transform(z, svh) -> np.ndarray:
    """y = H(z) * 2^-3 * svh (TensorFold PR, "Arithmetic" step 3)."""
    return blockwise_hadamard(z) * 2.0 ** -3 * np.asarray(svh, dtype=np.float64)


def _shard_of_block(shard_cols: Sequence[int], c: int) -> int:
    for s in range(len(shard_cols) - 1):
        if shard_cols[s] <= 128 * c < shard_cols[s + 1]:
            return s
    raise ValueError("column block outside the layer")


def linear_dense(x, w, suh, svh, shard_cols: Sequence[int]) -> np.ndarray:
    """The layer with an explicit dense Wq [K, N]; each shard feeds its own columns."""
    xh = input_transform(x, suh)
    w = np.asarray(w, dtype=np.float64)
    z = np.zeros((xh.shape[1], w.shape[1]))
    for s in range(len(shard_cols) - 1):
        a, b = shard_cols[s], shard_cols[s + 1]
        z[:, a:b] = xh[s] @ w[:, a:b]
    return output_transform(z, svh)


def linear(x, trellis, bits: int, cb: int, suh, svh, shard_cols: Sequence[int],
           col_blocks: Optional[Sequence[int]] = None) -> np.ndarray:
    """y (float64) of the layer, optionally only for selected 128-column blocks.

    Wq is decoded one 128-column block at a time so that wide layers never
    materialise a full float64 weight matrix.  Rows are independent, so a
    caller may pass any subset of rows of x.
    """
    x = np.asarray(x, dtype=np.float64)
    suh = np.atleast_2d(np.asarray(suh, dtype=np.float64))
    svh = np.asarray(svh, dtype=np.float64)
    n = shard_cols[-1]
    blocks = list(range(n // 128)) if col_blocks is None else list(col_blocks)
    xh = input_transform(x, suh)
    out = np.zeros((x.shape[0], 128 * len(blocks)))
    for i, c in enumerate(blocks):
        w = dequantize(trellis, bits, cb, [c])
        z = xh[_shard_of_block(shard_cols, c)] @ w
        out[:, 128 * i:128 * i + 128] = output_transform(z, svh[128 * c:128 * c + 128])
    return out


def linear_bruteforce(x, trellis, bits: int, cb: int, suh, svh, shard_cols: Sequence[int]) -> np.ndarray:
    """Naive loops from the bit-serial unpacker; tiny K, N only.

    Every sum is written out term by term, the Hadamard entries come from
    the popcount definition, and the weights from ``trellis_states_bitserial``.
    """
    x = np.asarray(x, dtype=np.float64)
    suh = np.atleast_2d(np.asarray(suh, dtype=np.float64))
    svh = np.asarray(svh, dtype=np.float64)
    tr = np.asarray(trellis)
    m, k = x.shape
    n = shard_cols[-1]

    def had(i: int, j: int) -> float:
        return -1.0 if bin(i & j).count("1") % 2 else 1.0

    wq = np.zeros((k, n))
    for kt in range(k // 16):
        for nt in range(n // 16):
            st = trellis_states_bitserial(tr[kt, nt], bits)
            vals = half_bits_to_f64(codebook(cb, st))
            for v in range(256):
                lk, ln = tile_position(v)
                wq[16 * kt + lk, 16 * nt + ln] = vals[v]
    y = np.zeros((m, n))
    for r in range(m):
        for s in range(len(shard_cols) - 1):
            xr = np.zeros(k)
            for blk in range(k // 128):
                for i in range(128):
                    acc = 0.0
                    for j in range(128):
                        acc += had(i, j) * x[r, 128 * blk + j] * suh[s, 128 * blk + j]
                    xr[128 * blk + i] = acc / 16.0
            for col in range(shard_cols[s], shard_cols[s + 1]):
                acc = 0.0
                for kk in range(k):
                    acc += xr[kk] * wq[kk, col]
                y[r, col] = acc
        z = y[r].copy()
        for blk in range(n // 128):
            for i in range(128):
                acc = 0.0
                for j in range(128):
                    acc += had(i, j) * z[128 * blk + j]
                y[r, 128 * blk + i] = acc / 8.0 * svh[128 * blk + i]
    return y


# ---------------------------------------------------------------------------
# Mixture of experts (cuda-exl3 README, "What is supported": routed experts run
# as a grouped GEMM over block-aligned (token, expert) pairs, the trellis offset
# by a per-block expert id; exl3_moe_had_in gathers each routed row and rotates
# it with its own expert's suh; "MoE notes": blocks of no expert carry -1 and
# are skipped)
# ---------------------------------------------------------------------------


def _routed_token(sorted_ids, r: int, num_tokens: int, topk: int) -> int:
    """Token of padded row r, or -1 for a padding row."""
    i = int(sorted_ids[r])
    return i // topk if 0 <= i < num_tokens * topk else -1


def moe_input_transform(x, sorted_ids, block_expert, block: int, topk: int, suh) -> np.ndarray:
    """xh[s, r] = the input transform of row r's token with its block's expert's
    suh (float64 [S, rows, K]); padding rows and rows of -1 blocks are zero."""
    x = np.asarray(x, dtype=np.float64)
    suh = np.asarray(suh, dtype=np.float64)  # [E, S, K]
    rows = len(sorted_ids)
    xh = np.zeros((suh.shape[1], rows, x.shape[1]))
    for b, e in enumerate(np.asarray(block_expert)):
        if e < 0:
            continue
        for r in range(b * block, (b + 1) * block):
            t = _routed_token(sorted_ids, r, x.shape[0], topk)
            if t >= 0:
                xh[:, r] = input_transform(x[t][None], suh[e])[:, 0]
    return xh


def moe_linear(x, sorted_ids, block_expert, block: int, topk: int, trellis, bits: int, cb: int, suh, svh,
               shard_cols: Sequence[int]) -> np.ndarray:
    """Rows of the grouped GEMM, float64 [rows, N]: row r is its token's output
    through its block's expert (the layer with that expert's trellis, suh and
    svh); padding rows are 0 and rows of -1 blocks NaN (never written)."""
    x = np.asarray(x, dtype=np.float64)
    rows = len(sorted_ids)
    n = shard_cols[-1]
    y = np.full((rows, n), np.nan)
    for b, e in enumerate(np.asarray(block_expert)):
        if e < 0:
            continue
        toks = [_routed_token(sorted_ids, r, x.shape[0], topk) for r in range(b * block, (b + 1) * block)]
        xb = np.stack([x[t] if t >= 0 else np.zeros(x.shape[1]) for t in toks])
        y[b * block:(b + 1) * block] = linear(xb, np.asarray(trellis[e]), bits, cb, np.asarray(suh[e]),
                                              np.asarray(svh[e]), shard_cols)
    return y


def moe_combine(y_rows, sorted_ids, block_expert, block: int, topk: int, weights, num_tokens: int,
                num_experts: int) -> np.ndarray:
    """The weighted combine of each token's top-k expert outputs, float64
    [num_tokens, N].

    Reading (the pages run the routed experts as a grouped GEMM over
    block-aligned rows and leave the combine to the caller: cuda-exl3 README,
    "What is supported", "MoE notes"): out[t] = sum over the slots s of token
    t, in ascending s, of weights[t, s] * y_rows[r], where r is the padded row
    of a live block (expert id in [0, num_experts)) whose sorted_ids entry is
    the pair t * topk + s.  A pair with no such row adds nothing; padding rows
    and rows of blocks of no expert are never read."""
    y = np.asarray(y_rows, dtype=np.float64)
    w = np.asarray(weights, dtype=np.float64).reshape(num_tokens, topk)
    ids = np.asarray(sorted_ids)
    experts = np.asarray(block_expert)
    row_of = {}
    for r in range(len(ids)):
        e = int(experts[r // block])
        p = int(ids[r])
        if 0 <= e < num_experts and 0 <= p < num_tokens * topk:
            row_of[p] = r
    out = np.zeros((num_tokens, y.shape[1]))
    for t in range(num_tokens):
        for s in range(topk):
            r = row_of.get(t * topk + s)
            if r is not None:
                out[t] += w[t, s] * y[r]
    return out
