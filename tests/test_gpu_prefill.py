"""GPU parity of the chunkwise prefill against the float64 token-by-token oracle, through the
C ABI: varlen packing with ragged tails, continuation from a slot's state, the full-size
T=4096 single sequence (sampled by K-heads), and prefill followed by decode."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_09_gb300 import gdn, synth
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


def _dev_i32(x):
    return torch.from_numpy(np.asarray(x, np.int32)).cuda()


@pytest.mark.parametrize("geo", [
    synth.Geometry(2, 4, 128, 128, 4, synth.BF16),
    synth.Geometry(2, 2, 64, 64, 4, synth.F32),
    synth.Geometry(1, 3, 128, 64, 4, synth.BF16),
    synth.Geometry(2, 4, 64, 128, 4, synth.F32),
    synth.Geometry(2, 4, 128, 128, 4, synth.F32),
    synth.Geometry(1, 3, 128, 128, 4, synth.BF16),
    synth.Geometry(1, 4, 128, 128, 4, synth.BF16),   # four V-heads per K-head: the tensor-core path's limit
    synth.Geometry(1, 6, 64, 64, 4, synth.F32),      # six: the CUDA-core kernels
], ids=lambda g: f"Hk{g.Hk}Hv{g.Hv}dk{g.dk}dv{g.dv}{g.act}")
def test_prefill_varlen_full_compare(geo):
    lens = [1, 63, 0, 64, 65, 130, 2, 200]
    has_init = np.array([0, 1, 1, 0, 1, 0, 1, 1], np.uint8)
    n = len(lens)
    N = n + 3
    w = synth.make_weights(geo, 600)
    rec, conv = synth.make_pool(geo, N, 601, True)
    layer = GatedDeltaNetLayer(geo, w, N)
    layer.load_state(rec, conv)
    cu = synth.cu_seqlens(lens)
    slots = np.array([9, 0, 4, 2, 10, 5, 1, 7], np.int32)
    xs = synth.make_token_inputs(geo, int(cu[-1]), 602)
    out = layer.prefill(_dev_i32(cu), _dev_i32(slots), torch.from_numpy(has_init).cuda(),
                        **layer.inputs(xs))
    r64, c64 = rec.astype(np.float64), conv.astype(np.float64)
    rc, ref = oracle.prefill(geo.oracle_dims(), f64(w), r64, c64, cu, slots, has_init, **f64(xs))
    assert rc == 0
    torch.cuda.synchronize()
    assert_out_close(_np(out), ref, geo.act, "prefill outputs")
    g_rec, g_conv = _np(layer.rec_state), _np(layer.conv_state)
    for s in slots:
        assert_state_close(g_rec[s], r64[s], f"slot {s}")
        np.testing.assert_array_equal(g_conv[s], c64[s])
    for s in (3, 6, 8):
        np.testing.assert_array_equal(g_rec[s], rec[s])
        np.testing.assert_array_equal(g_conv[s], conv[s])
    assert int(layer.status.item()) == 0


def test_prefill_full_size_T4096_sampled_heads():
    wl = synth.workloads()[3]
    geo = wl.geo
    w = synth.make_weights(geo, wl.seed)
    layer = GatedDeltaNetLayer(geo, w, wl.num_slots)
    cu = synth.cu_seqlens(wl.seq_lens)
    T = int(cu[-1])
    xs = synth.make_token_inputs(geo, T, wl.seed, 0)
    slots = np.array([0], np.int32)
    out = layer.prefill(_dev_i32(cu), _dev_i32(slots), None, **layer.inputs(xs))
    torch.cuda.synchronize()
    got = _np(out)
    g_rec = _np(layer.rec_state)
    g_conv = _np(layer.conv_state)
    for k_heads in ([0], [7, 15]):
        hs = HeadSlice(geo, k_heads)
        r64 = np.zeros((1, hs.sub.Hv, geo.dk, geo.dv))
        c64 = np.zeros((1, geo.K - 1, hs.sub.cqkv))
        rc, ref = oracle.prefill(hs.sub.oracle_dims(), hs.weights(w), r64, c64, cu, slots, None,
                                 **hs.inputs(xs))
        assert rc == 0
        assert_out_close(hs.out_cols(got), ref, geo.act, f"heads {k_heads}")
        assert_state_close(hs.rec(g_rec)[0], r64[0], f"final state heads {k_heads}")
        np.testing.assert_array_equal(hs.conv(g_conv)[0], c64[0])


def test_prefill_pipelined_windows_four_sequences():
    """Four sequences at the production geometry (Hk=16, Hv=32, d=128): their 128 chains leave
    SMs free, so the call runs in pipelined windows whose chunks span sequence boundaries; one
    sequence continues from its slot.  Sampled K-heads against the oracle, every touched slot's
    state and conv state, and an untouched slot left alone."""
    geo = synth.Geometry(16, 32, 128, 128, 4, synth.BF16)
    w = synth.make_weights(geo, 620)
    lens = [700, 130, 1500, 64]
    cu = synth.cu_seqlens(lens)
    T = int(cu[-1])
    xs = synth.make_token_inputs(geo, T, 621, 0)
    rec0, conv0 = synth.make_pool(geo, 6, 622, True)
    layer = GatedDeltaNetLayer(geo, w, 6)
    layer.load_state(rec0, conv0)
    slots = np.array([4, 1, 0, 3], np.int32)
    has_init = np.array([0, 1, 0, 0], np.uint8)
    before = layer.rec_state[5].clone()
    out = layer.prefill(_dev_i32(cu), _dev_i32(slots),
                        torch.from_numpy(has_init).cuda(), **layer.inputs(xs))
    torch.cuda.synchronize()
    got = _np(out)
    g_rec = _np(layer.rec_state)
    g_conv = _np(layer.conv_state)
    assert torch.equal(layer.rec_state[5], before)
    for k_heads in ([3], [10, 15]):
        hs = HeadSlice(geo, k_heads)
        r64 = hs.rec(rec0)
        c64 = hs.conv(conv0)
        rc, ref = oracle.prefill(hs.sub.oracle_dims(), hs.weights(w), r64, c64, cu, slots, has_init,
                                 **hs.inputs(xs))
        assert rc == 0
        assert_out_close(hs.out_cols(got), ref, geo.act, f"heads {k_heads}")
        for sl in slots:
            assert_state_close(hs.rec(g_rec)[sl], r64[sl], f"slot {sl} heads {k_heads}")
            np.testing.assert_array_equal(hs.conv(g_conv)[sl], c64[sl])
    assert int(layer.status.item()) == 0


def test_prefill_then_decode_continues():
    geo = synth.Geometry(2, 4, 128, 128, 4, synth.BF16)
    w = synth.make_weights(geo, 610)
    T = 150
    xs = synth.make_token_inputs(geo, T + 1, 611)
    layer = GatedDeltaNetLayer(geo, w, 3)
    head = {k: v[:T] for k, v in xs.items()}
    tail = {k: v[T:] for k, v in xs.items()}
    layer.prefill(_dev_i32([0, T]), _dev_i32([2]), None, **layer.inputs(head))
    out = layer.decode_step(_dev_i32([2]), **layer.inputs(tail))
    r64 = np.zeros((3, geo.Hv, geo.dk, geo.dv))
    c64 = np.zeros((3, geo.K - 1, geo.cqkv))
    _, ref = oracle.prefill(geo.oracle_dims(), f64(w), r64, c64, [0, T + 1], [2], None, **f64(xs))
    torch.cuda.synchronize()
    assert_out_close(_np(out), ref[T:], geo.act, "decode after prefill")
    assert_state_close(_np(layer.rec_state)[2], r64[2], "state")
    np.testing.assert_array_equal(_np(layer.conv_state)[2], c64[2])


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_bad_slot_and_bad_seqlens(d):
    geo = synth.Geometry(1, 2, d, d, 4, synth.BF16)
    w = synth.make_weights(geo, 620)
    rec, conv = synth.make_pool(geo, 2, 621, True)
    layer = GatedDeltaNetLayer(geo, w, 2)
    layer.load_state(rec, conv)
    xs = synth.make_token_inputs(geo, 70, 622)
    out = layer.prefill(_dev_i32([0, 30, 70]), _dev_i32([5, 1]), None, **layer.inputs(xs))
    torch.cuda.synchronize()
    assert int(layer.status.item()) & 1
    got = _np(out)
    assert np.all(got[:30] == 0.0)
    np.testing.assert_array_equal(_np(layer.rec_state)[0], rec[0])
    r64, c64 = rec.astype(np.float64), conv.astype(np.float64)
    _, ref = oracle.prefill(geo.oracle_dims(), f64(w), r64, c64, [0, 30, 70], [5, 1], None,
                            **f64(xs))
    assert_out_close(got[30:], ref[30:], geo.act)
    # decreasing cu_seqlens: reported on the status word, nothing written
    layer.status.zero_()
    layer.load_state(rec, conv)
    sentinel = torch.full((70, geo.zdim), 7.0, dtype=torch.bfloat16, device="cuda")
    layer.prefill(_dev_i32([0, 50, 40]), _dev_i32([0, 1]), None, out=sentinel, **layer.inputs(xs))
    torch.cuda.synchronize()
    assert int(layer.status.item()) & 2
    assert torch.all(sentinel == 7.0)
    np.testing.assert_array_equal(_np(layer.rec_state), rec)


def test_prefill_many_short_sequences():
    """257 sequences of 0..70 tokens (most shorter than one chunk), mixed initial states, on the
    tensor-core path (d = 128): every output and state against the oracle."""
    geo = synth.Geometry(2, 4, 128, 128, 4, synth.BF16)
    rng = np.random.default_rng(640)
    n = 257
    lens = [int(x) for x in rng.integers(0, 71, n)]
    has_init = rng.integers(0, 2, n).astype(np.uint8)
    N = n + 5
    w = synth.make_weights(geo, 641)
    rec, conv = synth.make_pool(geo, N, 642, True)
    layer = GatedDeltaNetLayer(geo, w, N)
    layer.load_state(rec, conv)
    cu = synth.cu_seqlens(lens)
    slots = rng.permutation(N)[:n].astype(np.int32)
    xs = synth.make_token_inputs(geo, int(cu[-1]), 643)
    out = layer.prefill(_dev_i32(cu), _dev_i32(slots), torch.from_numpy(has_init).cuda(),
                        **layer.inputs(xs))
    r64, c64 = rec.astype(np.float64), conv.astype(np.float64)
    rc, ref = oracle.prefill(geo.oracle_dims(), f64(w), r64, c64, cu, slots, has_init, **f64(xs))
    assert rc == 0
    torch.cuda.synchronize()
    assert_out_close(_np(out), ref, geo.act, "prefill outputs")
    g_rec, g_conv = _np(layer.rec_state), _np(layer.conv_state)
    for s in slots:
        assert_state_close(g_rec[s], r64[s], f"slot {s}")
        np.testing.assert_array_equal(g_conv[s], c64[s])
    untouched = sorted(set(range(N)) - set(slots.tolist()))
    for s in untouched:
        np.testing.assert_array_equal(g_rec[s], rec[s])
    assert int(layer.status.item()) == 0


def test_prefill_long_sequence_state_accuracy():
    """One 16384-token sequence (256 dependent chunk steps of the split-bf16 tensor-core chain)
    at the full head count, continuing from a pre-filled slot: outputs and the final state of
    two K-heads (with their V-heads) against the oracle."""
    wl = synth.workloads()[3]
    geo = wl.geo
    T = 16384
    w = synth.make_weights(geo, 660)
    rec, conv = synth.make_pool(geo, 2, 662, True)
    layer = GatedDeltaNetLayer(geo, w, 2)
    layer.load_state(rec, conv)
    xs = synth.make_token_inputs(geo, T, 661)
    cu = np.array([0, T], np.int32)
    slots = np.array([1], np.int32)
    has_init = np.array([1], np.uint8)
    out = layer.prefill(_dev_i32(cu), _dev_i32(slots), torch.from_numpy(has_init).cuda(),
                        **layer.inputs(xs))
    torch.cuda.synchronize()
    got = _np(out)
    g_rec, g_conv = _np(layer.rec_state), _np(layer.conv_state)
    for k_heads in ([5], [12]):
        hs = HeadSlice(geo, k_heads)
        r64 = hs.rec(rec).astype(np.float64)
        c64 = hs.conv(conv).astype(np.float64)
        rc, ref = oracle.prefill(hs.sub.oracle_dims(), hs.weights(w), r64, c64, cu, slots,
                                 has_init, **hs.inputs(xs))
        assert rc == 0
        assert_out_close(hs.out_cols(got), ref, geo.act, f"heads {k_heads}")
        assert_state_close(hs.rec(g_rec)[1], r64[1], f"final state heads {k_heads}")
        np.testing.assert_array_equal(hs.conv(g_conv)[1], c64[1])


def _varlen_case(geo, seed):
    lens = [1, 63, 0, 64, 65, 130, 2, 200, 129]
    has_init = np.array([0, 1, 1, 0, 1, 0, 1, 1, 0], np.uint8)
    n = len(lens)
    N = n + 3
    w = synth.make_weights(geo, seed)
    rec, conv = synth.make_pool(geo, N, seed + 1, True)
    cu = synth.cu_seqlens(lens)
    slots = np.array([9, 0, 4, 2, 10, 5, 1, 7, 11], np.int32)
    xs = synth.make_token_inputs(geo, int(cu[-1]), seed + 2)
    return w, rec, conv, cu, slots, has_init, xs, N


@pytest.mark.parametrize("cap_chunks,geo", [
    (1, synth.Geometry(2, 4, 128, 128, 4, synth.BF16)),
    (2, synth.Geometry(2, 4, 128, 128, 4, synth.BF16)),
    (5, synth.Geometry(2, 4, 128, 128, 4, synth.BF16)),
    (2, synth.Geometry(2, 2, 128, 128, 4, synth.F32)),
    (3, synth.Geometry(1, 3, 128, 128, 4, synth.BF16)),
], ids=lambda x: f"{x.Hk}x{x.Hv}{x.act}" if isinstance(x, synth.Geometry) else f"cap{x}")
def test_prefill_windowed_workspace(cap_chunks, geo):
    """A workspace of only `cap_chunks` chunks' records: the call runs in windows of whole chunks
    (sequences cross window edges, an empty sequence, mixed initial states).  Outputs and states
    against the oracle, and bit-equal to the same call with the full workspace."""
    w, rec, conv, cu, slots, has_init, xs, N = _varlen_case(geo, 670)
    full = GatedDeltaNetLayer(geo, w, N)
    capd = GatedDeltaNetLayer(geo, w, N)
    one = gdn.gdn_prefill_workspace_bytes(capd.dims, 1, 1)
    capd.ws_cap = cap_chunks * one
    assert gdn.gdn_prefill_workspace_bytes(capd.dims, len(slots), int(cu[-1])) > capd.ws_cap
    outs = []
    for layer in (full, capd):
        layer.load_state(rec, conv)
        outs.append(layer.prefill(_dev_i32(cu), _dev_i32(slots), torch.from_numpy(has_init).cuda(),
                                  **layer.inputs(xs)))
    torch.cuda.synchronize()
    assert capd._ws[:capd.ws_cap].numel() == capd.ws_cap
    r64, c64 = rec.astype(np.float64), conv.astype(np.float64)
    rc, ref = oracle.prefill(geo.oracle_dims(), f64(w), r64, c64, cu, slots, has_init, **f64(xs))
    assert rc == 0
    assert_out_close(_np(outs[1]), ref, geo.act, "windowed prefill outputs")
    g_rec, g_conv = _np(capd.rec_state), _np(capd.conv_state)
    for s in slots:
        assert_state_close(g_rec[s], r64[s], f"slot {s}")
        np.testing.assert_array_equal(g_conv[s], c64[s])
    for s in (3, 6, 8):
        np.testing.assert_array_equal(g_rec[s], rec[s])
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(full.rec_state, capd.rec_state)
    assert torch.equal(full.conv_state, capd.conv_state)
    assert int(capd.status.item()) == 0


def test_prefill_65536_tokens_bounded_workspace():
    """One 65,536-token sequence at the full head count (Hk=16, Hv=32, d=128) with the workspace
    capped at 256 MiB (the single-window size would be 4.85 GB): outputs and final state of one
    K-head (and its two V-heads) against the oracle."""
    geo = synth.workloads()[3].geo
    T = 65536
    w = synth.make_weights(geo, 680)
    layer = GatedDeltaNetLayer(geo, w, 1)
    layer.ws_cap = 256 << 20
    assert gdn.gdn_prefill_workspace_bytes(layer.dims, 1, T) > 4 * layer.ws_cap
    xs = synth.make_token_inputs(geo, T, 681)
    cu = np.array([0, T], np.int32)
    slots = np.array([0], np.int32)
    out = layer.prefill(_dev_i32(cu), _dev_i32(slots), None, **layer.inputs(xs))
    torch.cuda.synchronize()
    assert layer._ws.numel() <= layer.ws_cap
    got = _np(out)
    g_rec, g_conv = _np(layer.rec_state), _np(layer.conv_state)
    hs = HeadSlice(geo, [9])
    r64 = np.zeros((1, hs.sub.Hv, geo.dk, geo.dv))
    c64 = np.zeros((1, geo.K - 1, hs.sub.cqkv))
    rc, ref = oracle.prefill(hs.sub.oracle_dims(), hs.weights(w), r64, c64, cu, slots, None,
                             **hs.inputs(xs))
    assert rc == 0
    assert_out_close(hs.out_cols(got), ref, geo.act, "65,536-token outputs, K-head 9")
    assert_state_close(hs.rec(g_rec)[0], r64[0], "65,536-token final state, K-head 9")
    np.testing.assert_array_equal(hs.conv(g_conv)[0], c64[0])
    assert int(layer.status.item()) == 0


def test_concurrent_prefill_calls_on_two_streams():
    """Two prefill calls over disjoint slots, each with its own workspace, issued from two host
    threads on two streams at once, equal the same calls made one after another."""
    import threading
    geo = synth.Geometry(2, 4, 128, 128, 4, synth.BF16)
    w = synth.make_weights(geo, 640)
    rec0, conv0 = synth.make_pool(geo, 6, 641, True)
    layer = GatedDeltaNetLayer(geo, w, 6)
    calls = []
    for j, (lens, slots, init) in enumerate((([300, 77], [0, 3], [1, 0]), ([450], [5], [0]))):
        cu = synth.cu_seqlens(lens)
        xs = layer.inputs(synth.make_token_inputs(geo, int(cu[-1]), 642 + j, 0))
        calls.append((_dev_i32(cu), _dev_i32(slots), torch.tensor(init, dtype=torch.uint8, device="cuda"),
                      len(lens), int(cu[-1]), xs))
    # one after another
    layer.load_state(rec0, conv0)
    seq = [_np(layer.prefill(cu, sl, hi, **xs)) for cu, sl, hi, n, T, xs in calls]
    torch.cuda.synchronize()
    seq_rec, seq_conv = _np(layer.rec_state).copy(), _np(layer.conv_state).copy()
    # at once, one thread and one stream per call, each with its own workspace
    layer.load_state(rec0, conv0)
    outs = [torch.empty((T, geo.zdim), dtype=torch.bfloat16, device="cuda") for _, _, _, _, T, _ in calls]
    wss = [torch.empty(max(gdn.gdn_prefill_workspace_bytes(layer.dims, n, T), 256), dtype=torch.uint8,
                       device="cuda") for _, _, _, n, T, _ in calls]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    errors = []

    def run(j):
        try:
            cu, sl, hi, n, T, xs = calls[j]
            with torch.cuda.stream(streams[j]):
                gdn.gdn_prefill_chunked(layer.dims, layer.w, layer.pool, cu, sl, hi, n, T, xs["qkv"],
                                        xs["z"], xs["a"], xs["b"], outs[j], wss[j], streams[j])
        except Exception as e:   # reported below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(j,)) for j in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for j in range(2):
        np.testing.assert_array_equal(_np(outs[j]), seq[j])
    np.testing.assert_array_equal(_np(layer.rec_state), seq_rec)
    np.testing.assert_array_equal(_np(layer.conv_state), seq_conv)
    assert int(layer.status.item()) == 0
