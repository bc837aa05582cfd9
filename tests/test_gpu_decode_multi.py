"""GPU parity of the multi-token decode (T consecutive tokens per row, one state read and write)
against the float64 oracle run as T successive single-token decode steps, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_09_gb300 import synth
from gated_deltanet_linear_09_gb300.runtime import GatedDeltaNetLayer
from gpu_util import HeadSlice, assert_out_close, assert_state_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_linear_09_gb300 import build, gdn
    build.build()
    gdn.load()


def _np(t):
    return t.detach().float().cpu().numpy()


def _layer(geo, seed, num_slots, prefilled):
    w = synth.make_weights(geo, seed)
    rec, conv = synth.make_pool(geo, num_slots, seed, prefilled)
    layer = GatedDeltaNetLayer(geo, w, num_slots)
    layer.load_state(rec, conv)
    return layer, w, rec, conv


def _multi_inputs(geo, B, T, seed, step):
    """[B][T][...] inputs: token t of every row drawn like a decode step's inputs."""
    toks = [synth.make_token_inputs(geo, B, seed, step, t) for t in range(T)]
    return {k: np.stack([x[k] for x in toks], axis=1) for k in toks[0]}


def _oracle_multi(geo, w64, r64, c64, slots, xs):
    """T successive single-token oracle decode steps; outputs [B][T][Hv*dv]."""
    T = next(iter(xs.values())).shape[1]
    outs = []
    for t in range(T):
        rc, o = oracle.decode_step(geo.oracle_dims(), w64, r64, c64, slots,
                                   **{k: np.asarray(v[:, t], np.float64) for k, v in xs.items()})
        assert rc == 0
        outs.append(o)
    return np.stack(outs, axis=1)


@pytest.mark.parametrize("T", [1, 2, 5, 8])
@pytest.mark.parametrize("geo", [
    synth.Geometry(2, 6, 128, 128, 4, synth.BF16),
    synth.Geometry(2, 4, 64, 64, 4, synth.F32),
    synth.Geometry(3, 3, 128, 64, 4, synth.BF16),
    synth.Geometry(1, 4, 64, 128, 4, synth.F32),
], ids=lambda g: f"Hk{g.Hk}Hv{g.Hv}dk{g.dk}dv{g.dv}{g.act}")
def test_decode_multi_full_compare(geo, T):
    """Every output and state over 3 calls of T tokens, a padding row, untouched slots."""
    N = 6
    layer, w, rec, conv = _layer(geo, 700 + T, N, True)
    slots = np.array([4, -1, 0, 2], np.int32)
    sl_dev = torch.from_numpy(slots).cuda()
    w64 = f64(w)
    r64, c64 = rec.astype(np.float64), conv.astype(np.float64)
    for step in range(3):
        xs = _multi_inputs(geo, len(slots), T, 701, step)
        out = layer.decode_multi(sl_dev, **layer.inputs(xs))
        ref = _oracle_multi(geo, w64, r64, c64, slots, xs)
        got = _np(out)
        assert got.shape == (len(slots), T, geo.zdim)
        assert_out_close(got, ref, geo.act, f"call {step}")
        assert np.all(got[1] == 0.0)
    torch.cuda.synchronize()
    g_rec, g_conv = _np(layer.rec_state), _np(layer.conv_state)
    for s in (4, 0, 2):
        assert_state_close(g_rec[s], r64[s], f"slot {s}")
        np.testing.assert_array_equal(g_conv[s], c64[s])
    for s in (1, 3, 5):
        np.testing.assert_array_equal(g_rec[s], rec[s])
        np.testing.assert_array_equal(g_conv[s], conv[s])
    assert int(layer.status.item()) == 0


def test_decode_multi_matches_single_steps_on_gpu():
    """T tokens in one call and T single-token calls land on the same state (both are checked
    against the oracle above); here the two GPU paths are compared with each other."""
    geo = synth.Geometry(2, 4, 128, 128, 4, synth.BF16)
    T = 4
    la, w, rec, conv = _layer(geo, 720, 3, True)
    lb = GatedDeltaNetLayer(geo, w, 3)
    lb.load_state(rec, conv)
    slots = torch.tensor([2, 0], dtype=torch.int32, device="cuda")
    xs = _multi_inputs(geo, 2, T, 721, 0)
    out_m = _np(la.decode_multi(slots, **la.inputs(xs)))
    for t in range(T):
        o = lb.decode_step(slots, **lb.inputs({k: np.ascontiguousarray(v[:, t]) for k, v in xs.items()}))
        np.testing.assert_allclose(out_m[:, t], _np(o), rtol=0, atol=8e-3)
    torch.cuda.synchronize()
    for s in (2, 0):
        assert_state_close(_np(la.rec_state)[s], _np(lb.rec_state)[s].astype(np.float64), f"slot {s}")
    np.testing.assert_array_equal(_np(la.conv_state), _np(lb.conv_state))


def test_decode_multi_full_size_sampled():
    """B=64 rows of 128 slots, Hk=16, Hv=48, d=128, T=4: the launch the bench times, checked on
    two K-heads (with their V-heads) of every row against the oracle."""
    wl = synth.workloads()[2]
    geo = wl.geo
    T = 4
    layer, w, rec, conv = _layer(geo, wl.seed, wl.num_slots, True)
    slots = synth.make_slot_idx(wl.num_slots, wl.batch, wl.seed)
    sl_dev = torch.from_numpy(slots).cuda()
    xs = _multi_inputs(geo, wl.batch, T, wl.seed, 0)
    out = _np(layer.decode_multi(sl_dev, **layer.inputs(xs)))
    torch.cuda.synchronize()
    hs = HeadSlice(geo, [0, 11])
    w64 = hs.weights(w)
    r64 = hs.rec(rec).astype(np.float64)
    c64 = hs.conv(conv).astype(np.float64)
    sx = {k: (np.asarray(v, np.float64)[..., hs.ch] if k == "qkv" else
              np.asarray(v, np.float64)[..., hs.zcol] if k == "z" else
              np.asarray(v, np.float64)[..., hs.v_heads]) for k, v in xs.items()}
    ref = _oracle_multi(hs.sub, w64, r64, c64, slots, sx)
    assert_out_close(out[..., hs.zcol], ref, geo.act, "sampled heads")
    g_rec = _np(layer.rec_state)
    for s in slots[:8]:
        assert_state_close(g_rec[s][hs.v_heads], r64[s], f"slot {s}")


def test_decode_multi_rejects_bad_token_count():
    from gated_deltanet_linear_09_gb300 import gdn
    geo = synth.Geometry(2, 4, 64, 64, 4, synth.F32)
    layer, w, rec, conv = _layer(geo, 730, 2, False)
    slots = torch.tensor([0], dtype=torch.int32, device="cuda")
    inp9 = layer.inputs(_multi_inputs(geo, 1, 9, 731, 0))
    for inp in (inp9, {k: v[:, :0].contiguous() for k, v in inp9.items()}):   # T = 9 and T = 0
        with pytest.raises(gdn.GdnError):
            layer.decode_multi(slots, **inp)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_np(layer.rec_state), rec)   # nothing launched


def test_decode_multi_captured_in_cuda_graph():
    """gdn_decode_multi is one launch with no host reads of device data: captured in a CUDA graph
    and replayed on refilled inputs, it matches eager calls bit for bit (outputs and state)."""
    geo = synth.Geometry(2, 6, 128, 128, 4, synth.BF16)
    T = 3
    la, w, rec, conv = _layer(geo, 730, 4, True)
    slots = torch.tensor([3, -1, 1], dtype=torch.int32, device="cuda")
    calls = [la.inputs(_multi_inputs(geo, 3, T, 731, c)) for c in range(3)]
    eager = [_np(la.decode_multi(slots, **x)) for x in calls]
    torch.cuda.synchronize()
    eager_state = _np(la.rec_state).copy()
    la.load_state(rec, conv)
    static = {k: torch.empty_like(v) for k, v in calls[0].items()}
    for k in static:
        static[k].copy_(calls[0][k])
    out = torch.empty((3, T, geo.zdim), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            la.decode_multi(slots, static["qkv"], static["z"], static["a"], static["b"], out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_np(la.rec_state), rec)   # capture runs nothing
    for x, ref in zip(calls, eager):
        for k in static:
            static[k].copy_(x[k])
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(_np(out), ref)
    np.testing.assert_array_equal(_np(la.rec_state), eager_state)
