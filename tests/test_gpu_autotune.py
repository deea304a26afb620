"""Tile-shape autotune (cuda-exl3 README, "Where the time goes"): the tile is
timed once per distinct layer shape and batch bucket, cached, and never tuned
while a CUDA graph is being captured.

Every tile shape computes the same bytes, so the tuned launch must equal the
cost model's launch byte for byte and meet the oracle's per-column bar; the
cache must hold one key per distinct call shape; a captured launch must neither
tune nor add a key.
"""
import pytest
import torch

import exl3_trellis_quantized_gb300 as E
from exl3_trellis_quantized_gb300 import synthetic
from oracle import exl3_oracle as O
from oracle_check import assert_columns

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _tuner_off():
    E.clear_autotune()
    yield
    E.set_autotune(False)
    E.clear_autotune()
    assert E.device_status() == 0


def _layer(k, cols, bits, cb, seed, host=False):
    layer = synthetic.make_layer(k, cols, bits, cb, seed=seed)
    dev = (layer.trellis.to(DEV), layer.suh.to(DEV), layer.svh.to(DEV), layer.shard_cols)
    return dev + (layer,) if host else dev


def _against_oracle(y, layer, m, m_case, seed):
    """The first m rows of the case's largest batch (m_case rows; make_x gives
    prefixes), against the oracle with the column max over that batch."""
    x = synthetic.make_x(m_case, layer.k, seed=seed)
    ref = O.linear(x.float().numpy(), layer.trellis.numpy(), layer.bits, layer.codebook,
                   layer.suh.float().numpy(), layer.svh.float().numpy(), layer.shard_cols)
    assert_columns(y.float().cpu().numpy(), ref[:m], "tuned launch", ref_batch=ref)


@pytest.mark.parametrize("m", [1, 16, 100, 300])
@pytest.mark.parametrize("bits,cb", [(2, 0), (4, 1), (6, 2)])
def test_tuned_equals_model(m, bits, cb):
    tr, suh, svh, cols, layer = _layer(1024, [512, 256], bits, cb, seed=7000 + bits, host=True)
    x = synthetic.make_x(m, 1024, seed=7001).to(DEV)
    xh = E.input_transform(x, suh)
    y_model = E.gemm(xh, tr, bits, cb, svh, cols)
    E.set_autotune(True)
    y_tuned = E.gemm(xh, tr, bits, cb, svh, cols)  # tunes, then launches the winner
    y_again = E.gemm(xh, tr, bits, cb, svh, cols)  # cached
    torch.cuda.synchronize()
    assert E.autotune_entries() == 1
    assert torch.equal(y_tuned.view(torch.int16), y_model.view(torch.int16))
    assert torch.equal(y_again.view(torch.int16), y_model.view(torch.int16))
    _against_oracle(y_tuned, layer, m, 300, 7001)


def test_split_k_tuned_equals_model():
    k, n, bits, cb, m = 4096, 256, 3, 1, 24
    tr, suh, svh, cols, layer = _layer(k, [n], bits, cb, seed=7100, host=True)
    parts = E.splitk_parts(k, n)
    assert parts > 1
    x = synthetic.make_x(m, k, seed=7101).to(DEV)
    xh = E.input_transform(x, suh)
    acc = torch.zeros(E.splitk_workspace_bytes(m, k, n) // 4, dtype=torch.float32, device=DEV)
    y_model = E.gemm_splitk(xh, tr, bits, cb, svh, cols, acc)
    E.set_autotune(True)
    y_tuned = E.gemm_splitk(xh, tr, bits, cb, svh, cols, acc)  # the trials rewrite the same partials
    torch.cuda.synchronize()
    assert E.autotune_entries() == 1
    assert torch.equal(y_tuned.view(torch.int16), y_model.view(torch.int16))
    assert not bool(acc.any()), "the epilogue leaves the workspace zeroed"
    _against_oracle(y_tuned, layer, m, m, 7101)


def test_keys_by_bucket_and_shape():
    tr, suh, svh, cols = _layer(512, [384], 4, 0, seed=7200)
    E.set_autotune(True)
    for m in (1, 7, 32):  # one bucket: m <= 32
        E.gemm(E.input_transform(synthetic.make_x(m, 512, seed=m).to(DEV), suh), tr, 4, 0, svh, cols)
    assert E.autotune_entries() == 1
    for m in (33, 64):  # bucket 64
        E.gemm(E.input_transform(synthetic.make_x(m, 512, seed=m).to(DEV), suh), tr, 4, 0, svh, cols)
    assert E.autotune_entries() == 2
    E.gemm(E.input_transform(synthetic.make_x(65, 512, seed=65).to(DEV), suh), tr, 4, 0, svh, cols)
    assert E.autotune_entries() == 3
    # another layer shape with the same batch gets its own key
    tr2, suh2, svh2, cols2 = _layer(512, [256], 4, 0, seed=7201)
    E.gemm(E.input_transform(synthetic.make_x(65, 512, seed=66).to(DEV), suh2), tr2, 4, 0, svh2, cols2)
    assert E.autotune_entries() == 4
    E.set_autotune(False)
    E.gemm(E.input_transform(synthetic.make_x(200, 512, seed=200).to(DEV), suh), tr, 4, 0, svh, cols)
    assert E.autotune_entries() == 4  # off: the model decides, nothing cached
    E.clear_autotune()
    assert E.autotune_entries() == 0


def _capture(fn):
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            fn()
    return graph


def test_no_tuning_under_graph_capture():
    k, m, bits, cb = 1024, 48, 5, 2
    tr, suh, svh, cols = _layer(k, [256, 256], bits, cb, seed=7300)
    x = synthetic.make_x(m, k, seed=7301).to(DEV)
    xh = E.input_transform(x, suh)
    y_model = E.gemm(xh, tr, bits, cb, svh, cols)
    E.set_autotune(True)
    y = torch.empty_like(y_model)
    graph = _capture(lambda: E.gemm(xh, tr, bits, cb, svh, cols, out=y))
    assert E.autotune_entries() == 0, "a captured launch must not tune"
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_model.view(torch.int16))


def test_eager_tuning_reaches_capture():
    """A key tuned eagerly is used, not re-tuned, by a captured launch."""
    k, m, bits, cb = 2048, 16, 3, 0
    tr, suh, svh, cols = _layer(k, [768], bits, cb, seed=7400)
    xh = E.input_transform(synthetic.make_x(m, k, seed=7401).to(DEV), suh)
    y_model = E.gemm(xh, tr, bits, cb, svh, cols)
    E.set_autotune(True)
    E.gemm(xh, tr, bits, cb, svh, cols)  # eager warm-up tunes the key
    assert E.autotune_entries() == 1
    y = torch.empty_like(y_model)
    graph = _capture(lambda: E.gemm(xh, tr, bits, cb, svh, cols, out=y))
    assert E.autotune_entries() == 1
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_model.view(torch.int16))
