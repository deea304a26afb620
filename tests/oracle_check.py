"""Shared comparison of GPU outputs with the oracle, used by the -m gpu tests.

The bar for a linear output is the layer specification's: per output column c,
|y_gpu[r, c] - y_oracle[r, c]| <= 4e-3 * max_r |y_oracle[r, c]|, the max taken
over the rows the case checks. A column whose reference is exactly zero (a pad)
must be exactly zero.

Every comparison also records err / (4e-3 * colmax), the fraction of the bar the
worst value used, under the running test's id; the conftest prints the largest
ones at the end of the session, so a kernel change that eats into the margin
shows up before it fails.
"""
import numpy as np

TOL = 4e-3
WORST = {}  # test id -> largest fraction of the bar used
_current = [None]


def oracle_linear(O, x, layer, col_blocks=None, trellis=None, suh=None, svh=None):
    """O.linear on a synthetic layer (optionally with replaced tensors), x a torch tensor or array."""
    xa = x.detach().float().cpu().numpy() if hasattr(x, "detach") else np.asarray(x, dtype=np.float64)
    tr = layer.trellis if trellis is None else trellis
    su = layer.suh if suh is None else suh
    sv = layer.svh if svh is None else svh
    return O.linear(xa, tr.numpy(), layer.bits, layer.codebook, su.float().numpy(), sv.float().numpy(),
                    layer.shard_cols, col_blocks=col_blocks)


def assert_columns(got, ref, what="", ref_batch=None):
    """Check got against ref column by column; returns the fraction of the bar used.

    ref_batch: the oracle's output for the case's largest batch, whose first rows
    are ref; the column max is taken over it (a small batch's rows are held to
    the bar of the batch they belong to, as every parity test does).
    """
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return 0.0
    colmax = np.abs(ref if ref_batch is None else np.asarray(ref_batch, dtype=np.float64)).max(axis=0)
    err = np.abs(got - ref)
    bad = err > TOL * colmax
    live = colmax > 0
    used = float(np.max(err[:, live] / (TOL * colmax[live]))) if live.any() else 0.0
    key = _current[0] or "?"
    WORST[key] = max(WORST.get(key, 0.0), used)
    assert not bad.any(), f"{what}: {bad.sum()} values out of tolerance, worst fraction of the bar {used:.3f}"
    return used
