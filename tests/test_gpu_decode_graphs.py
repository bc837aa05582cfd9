"""Bucketed CUDA-graph decode (gdn_decode_graphs_*): parity with the float64 oracle and bit
equality with eager gdn_decode_step calls, over steps whose batch size moves between buckets."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_09_gb300 import gdn, synth
from gated_deltanet_linear_09_gb300.runtime import DecodeGraphs, GatedDeltaNetLayer
from gpu_util import assert_out_close, assert_state_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_linear_09_gb300 import build
    build.build()
    gdn.load()


def _np(t):
    return t.detach().float().cpu().numpy()


def _write_rows(graphs, layer, slots, xs):
    B = len(slots)
    graphs.slot_idx[:B].copy_(torch.from_numpy(np.asarray(slots, np.int32)))
    dev = layer.inputs(xs)
    for k in ("qkv", "z", "a", "b"):
        getattr(graphs, k)[:B].copy_(dev[k])


@pytest.mark.parametrize("geo", [synth.Geometry(2, 4, 128, 128, 4, synth.BF16),
                                 synth.Geometry(2, 4, 64, 64, 4, synth.F32)],
                         ids=lambda g: f"d{g.dk}{g.act}")
def test_graph_decode_matches_oracle_and_eager(geo):
    N = 8
    w = synth.make_weights(geo, 800)
    rec, conv = synth.make_pool(geo, N, 800, True)
    lg = GatedDeltaNetLayer(geo, w, N)
    lg.load_state(rec, conv)
    le = GatedDeltaNetLayer(geo, w, N)
    le.load_state(rec, conv)
    graphs = DecodeGraphs(lg, [1, 2, 4, 8])
    assert graphs.max_batch == 8
    r64, c64 = rec.astype(np.float64), conv.astype(np.float64)
    rng = np.random.default_rng(801)
    for step, B in enumerate([3, 8, 1, 5, 2, 4, 7]):
        slots = rng.permutation(N)[:B].astype(np.int32)
        xs = synth.make_token_inputs(geo, B, 802, step)
        _write_rows(graphs, lg, slots, xs)
        got = graphs.step(B)
        bucket = min(b for b in (1, 2, 4, 8) if b >= B)
        eager = le.decode_step(torch.from_numpy(slots).cuda(), **le.inputs(xs))
        _, ref = oracle.decode_step(geo.oracle_dims(), f64(w), r64, c64, slots, **f64(xs))
        g = _np(got)
        assert_out_close(g, ref, geo.act, f"step {step}")
        np.testing.assert_array_equal(g, _np(eager))             # same kernel, same rows
        assert np.all(_np(graphs.out[B:bucket]) == 0.0)          # padding rows
    torch.cuda.synchronize()
    g_rec, g_conv = _np(lg.rec_state), _np(lg.conv_state)
    np.testing.assert_array_equal(g_rec, _np(le.rec_state))
    np.testing.assert_array_equal(g_conv, _np(le.conv_state))
    for s in range(N):
        assert_state_close(g_rec[s], r64[s], f"slot {s}")
        np.testing.assert_array_equal(g_conv[s], c64[s])
    assert int(lg.status.item()) == 0
    with pytest.raises(gdn.GdnError):
        graphs.step(9)                                           # above the largest bucket
    graphs.close()


def test_graph_create_rejects_bad_buckets():
    geo = synth.Geometry(2, 4, 64, 64, 4, synth.F32)
    layer = GatedDeltaNetLayer(geo, synth.make_weights(geo, 810), 2)
    for buckets in ([], [4, 2], [0, 1], [1, 1], list(range(1, 18))):
        with pytest.raises(gdn.GdnError):
            DecodeGraphs(layer, buckets)
