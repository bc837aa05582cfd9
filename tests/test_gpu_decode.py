"""GPU parity of the batched decode step, the standalone conv1d update and slot compaction
against the float64 oracle, through the C ABI (libgdn.so via the ctypes binding)."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_09_gb300 import synth
from gated_deltanet_linear_09_gb300.runtime import GatedDeltaNetLayer
from gpu_util import (HeadSlice, assert_out_close, assert_state_close, f64, rel_l2)

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


@pytest.mark.parametrize("geo", [
    synth.Geometry(2, 4, 64, 64, 4, synth.F32),
    synth.Geometry(2, 6, 128, 128, 4, synth.BF16),
    synth.Geometry(3, 3, 128, 64, 4, synth.BF16),
    synth.Geometry(1, 2, 64, 128, 4, synth.F32),
    synth.Geometry(1, 4, 128, 128, 4, synth.BF16),
    synth.Geometry(1, 6, 64, 64, 4, synth.F32),
], ids=lambda g: f"Hk{g.Hk}Hv{g.Hv}dk{g.dk}dv{g.dv}{g.act}")
def test_decode_small_full_compare(geo):
    """Every output, every state, padding rows and untouched slots, over 12 steps."""
    N, steps = 7, 12
    layer, w, rec, conv = _layer(geo, 500, N, True)
    slots = np.array([5, -1, 0, 3, 6], np.int32)          # one padding row
    sl_dev = torch.from_numpy(slots).cuda()
    ref_rec = rec.astype(np.float64)
    ref_conv = conv.astype(np.float64)
    for t in range(steps):
        xs = synth.make_token_inputs(geo, len(slots), 501, t)
        out = layer.decode_step(sl_dev, **layer.inputs(xs))
        rc, ref = oracle.decode_step(geo.oracle_dims(), f64(w), ref_rec, ref_conv, slots,
                                     **f64(xs))
        assert rc == 0
        got = _np(out)
        assert_out_close(got, ref, geo.act, f"step {t}")
        assert np.all(got[1] == 0.0)
    torch.cuda.synchronize()
    g_rec, g_conv = _np(layer.rec_state), _np(layer.conv_state)
    for s in (5, 0, 3, 6):
        assert_state_close(g_rec[s], ref_rec[s], f"slot {s}")
        np.testing.assert_array_equal(g_conv[s], ref_conv[s])
    for s in (1, 2, 4):                                     # untouched slots: bit-exact
        np.testing.assert_array_equal(g_rec[s], rec[s])
        np.testing.assert_array_equal(g_conv[s], conv[s])
    assert int(layer.status.item()) == 0


def test_decode_tiny_config_f32():
    """B=1, Hk=2, Hv=4, dk=dv=64, all f32, 16 steps from zero state."""
    wl = synth.workloads()[0]
    geo = wl.geo
    layer, w, rec, conv = _layer(geo, wl.seed, wl.num_slots, False)
    slots = synth.make_slot_idx(wl.num_slots, wl.batch, wl.seed)
    sl_dev = torch.from_numpy(slots).cuda()
    ref_rec, ref_conv = rec.astype(np.float64), conv.astype(np.float64)
    for t in range(wl.steps):
        xs = synth.decode_step_inputs(wl, t)
        out = layer.decode_step(sl_dev, **layer.inputs(xs))
        _, ref = oracle.decode_step(geo.oracle_dims(), f64(w), ref_rec, ref_conv, slots, **f64(xs))
        assert float(np.max(np.abs(_np(out) - ref))) <= 2e-3
        assert_state_close(_np(layer.rec_state), ref_rec, f"step {t}")
    np.testing.assert_array_equal(_np(layer.conv_state), ref_conv)


def test_decode_bad_slot_sets_status_and_skips_row():
    geo = synth.Geometry(2, 4, 128, 128, 4, synth.BF16)
    layer, w, rec, conv = _layer(geo, 510, 4, True)
    slots = np.array([1, 9, 2], np.int32)
    xs = synth.make_token_inputs(geo, 3, 511)
    out = layer.decode_step(torch.from_numpy(slots).cuda(), **layer.inputs(xs))
    torch.cuda.synchronize()
    assert int(layer.status.item()) & 1
    got = _np(out)
    assert np.all(got[1] == 0.0)
    ref_rec, ref_conv = rec.astype(np.float64), conv.astype(np.float64)
    rc, ref = oracle.decode_step(geo.oracle_dims(), f64(w), ref_rec, ref_conv, slots, **f64(xs))
    assert rc == -1
    assert_out_close(got, ref, geo.act)
    np.testing.assert_array_equal(_np(layer.rec_state)[[0, 3]], rec[[0, 3]])


def test_decode_row_permutation_and_determinism():
    geo = synth.Geometry(4, 8, 128, 128, 4, synth.BF16)
    layer, w, rec, conv = _layer(geo, 520, 12, True)
    slots = np.array([7, 2, 11, 0, 5, 9], np.int32)
    xs = synth.make_token_inputs(geo, 6, 521)
    dev = layer.inputs(xs)
    out1 = _np(layer.decode_step(torch.from_numpy(slots).cuda(), **dev))
    st1 = _np(layer.rec_state).copy()
    layer.load_state(rec, conv)
    perm = np.array([3, 5, 0, 1, 4, 2])
    dev_p = {k: v[torch.from_numpy(perm).cuda()].contiguous() for k, v in dev.items()}
    out2 = _np(layer.decode_step(torch.from_numpy(slots[perm]).cuda(), **dev_p))
    np.testing.assert_array_equal(out2, out1[perm])
    np.testing.assert_array_equal(_np(layer.rec_state), st1)
    layer.load_state(rec, conv)
    out3 = _np(layer.decode_step(torch.from_numpy(slots).cuda(), **dev))
    np.testing.assert_array_equal(out3, out1)                # run-to-run deterministic


def _run_decode_workload(wl, rows, k_heads, retire_at=None, n_retire=0):
    """Full-size decode workload on the GPU; the oracle follows sampled rows x K-heads."""
    geo = wl.geo
    layer, w, rec, conv = _layer(geo, wl.seed, wl.num_slots, wl.prefill_state)
    slots = synth.make_slot_idx(wl.num_slots, wl.batch, wl.seed)
    hs = HeadSlice(geo, k_heads)
    wsub = hs.weights(w)
    rows = list(rows)
    o_rec = np.ascontiguousarray(hs.rec(rec)[slots[rows]])      # oracle's private slots 0..n-1
    o_conv = np.ascontiguousarray(hs.conv(conv)[slots[rows]])
    o_slots = np.arange(len(rows), dtype=np.int32)
    cur_slots = slots.copy()
    B = wl.batch
    max_out_err = 0.0
    for t in range(wl.steps):
        if retire_at is not None and t == retire_at:
            torch.cuda.synchronize()
            retire = synth.retire_choice(wl.seed, B, n_retire, t)
            keep = np.array([i for i in range(B) if i not in set(retire.tolist())], np.int32)
            src = cur_slots[keep]
            dst = np.arange(len(keep), dtype=np.int32)
            before_r = layer.rec_state.clone()
            before_c = layer.conv_state.clone()
            layer.compact(src, dst)
            torch.cuda.synchronize()
            # compaction is a bit-exact snapshot gather; untouched slots keep their bytes
            exp_r = before_r.clone()
            exp_r[torch.from_numpy(dst).long().cuda()] = before_r[torch.from_numpy(src).long().cuda()]
            exp_c = before_c.clone()
            exp_c[torch.from_numpy(dst).long().cuda()] = before_c[torch.from_numpy(src).long().cuda()]
            assert torch.equal(layer.rec_state, exp_r)
            assert torch.equal(layer.conv_state, exp_c)
            # follow the sampled rows that survive
            newrow = {int(old): i for i, old in enumerate(keep)}
            surv = [j for j, r in enumerate(rows) if r in newrow]
            rows = [newrow[rows[j]] for j in surv]
            o_rec = np.ascontiguousarray(o_rec[surv])
            o_conv = np.ascontiguousarray(o_conv[surv])
            o_slots = np.arange(len(rows), dtype=np.int32)
            cur_slots = dst
            B = len(keep)
        sl_dev = torch.from_numpy(cur_slots).cuda()
        xs = synth.decode_step_inputs(wl, t, B)
        out = layer.decode_step(sl_dev, **layer.inputs(xs))
        if rows:
            _, ref = oracle.decode_step(hs.sub.oracle_dims(), wsub, o_rec, o_conv, o_slots,
                                        **hs.inputs(xs, rows))
            got = hs.out_cols(_np(out)[rows])
            max_out_err = max(max_out_err, assert_out_close(got, ref, geo.act, f"step {t}"))
        if t == 255 or t == wl.steps - 1:
            torch.cuda.synchronize()
            g = hs.rec(_np(layer.rec_state))[cur_slots[rows]]
            assert_state_close(g, o_rec, f"after step {t}")
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    return layer, max_out_err


def test_decode_batched_B16_256_steps():
    wl = synth.workloads()[1]
    _run_decode_workload(wl, rows=[0, 5, 15], k_heads=[0, 7, 15])


def test_decode_large_B64_512_steps_with_compaction():
    wl = synth.workloads()[2]
    _run_decode_workload(wl, rows=[0, 13, 31, 47, 63], k_heads=[0, 15], retire_at=256, n_retire=8)


def test_decode_production_geometry_f32_outputs():
    """The production head geometry (Hk=16, Hv=48, dk=dv=128, B=64 of 128 slots) in the f32
    activation mode, where the outputs carry no bf16 rounding: every sampled output within a bare
    2e-3 and the state within rel-L2 1e-4 after 256 steps."""
    base = synth.workloads()[2]
    wl = synth.Workload("decode_B64_Hk16_Hv48_d128_f32", synth.Geometry(16, 48, 128, 128, 4, synth.F32),
                        base.seed + 100, num_slots=128, batch=64, steps=256, prefill_state=True)
    _, mx = _run_decode_workload(wl, rows=[0, 21, 42, 63], k_heads=[0, 9, 15])
    assert mx <= 2e-3


# ------------------------------------------------------------------ conv1d and compaction

@pytest.mark.parametrize("act", [synth.F32, synth.BF16])
def test_conv1d_update_matches_oracle(act):
    geo = synth.Geometry(4, 8, 128, 128, 4, act)
    layer, w, rec, conv = _layer(geo, 530, 6, True)
    slots = np.array([4, -1, 1], np.int32)
    ref_conv = conv.astype(np.float64)
    for t in range(5):
        xs = synth.make_token_inputs(geo, 3, 531, t)
        qkv = layer.inputs(xs)["qkv"]
        out = layer.conv1d_update(torch.from_numpy(slots).cuda(), qkv)
        rc, ref = oracle.conv1d_update(np.asarray(w["conv_w"], np.float64), ref_conv, slots,
                                       np.asarray(xs["qkv"], np.float64))
        assert rc == 0
        assert_out_close(_np(out), ref, act, f"conv step {t}")
    np.testing.assert_array_equal(_np(layer.conv_state), ref_conv)


def test_compaction_bit_exact_overlap_and_cycles():
    geo = synth.Geometry(2, 4, 128, 128, 4, synth.BF16)
    layer, w, rec, conv = _layer(geo, 540, 10, True)
    cases = [
        ([7, 2, 9, 4, 0], [0, 1, 2, 3, 4]),      # gather into a prefix, overlapping
        ([0, 1, 2], [1, 2, 0]),                  # a 3-cycle
        ([3], [3]),                              # identity
        ([5, 5], [6, 8]),                        # one source, two destinations
    ]
    for src, dst in cases:
        before_r = _np(layer.rec_state).copy()
        before_c = layer.conv_state.clone()
        layer.compact(src, dst)
        torch.cuda.synchronize()
        exp_r = before_r.copy()
        exp_r[dst] = before_r[src]
        np.testing.assert_array_equal(_np(layer.rec_state), exp_r)
        exp_c = before_c.clone()
        exp_c[torch.tensor(dst).cuda()] = before_c[torch.tensor(src).cuda()]
        assert torch.equal(layer.conv_state, exp_c)
    # and the oracle's compaction agrees on the same lists
    r64, c64 = rec.astype(np.float64), conv.astype(np.float64)
    layer.load_state(rec, conv)
    for src, dst in cases:
        oracle.state_compact(r64, c64, np.array(src, np.int32), np.array(dst, np.int32))
        layer.compact(src, dst)
    np.testing.assert_array_equal(_np(layer.rec_state), r64.astype(np.float32))
    np.testing.assert_array_equal(_np(layer.conv_state), c64.astype(np.float32))


def test_compaction_many_pairs():
    geo = synth.Geometry(1, 1, 64, 64, 4, synth.F32)
    N = 3000
    layer, w, rec, conv = _layer(geo, 550, N, True)
    rng = np.random.default_rng(551)
    src = rng.permutation(N)[:2048].astype(np.int32)
    dst = rng.permutation(N)[:2048].astype(np.int32)
    before = _np(layer.rec_state).copy()
    layer.compact(src, dst)
    torch.cuda.synchronize()
    exp = before.copy()
    exp[dst] = before[src]
    np.testing.assert_array_equal(_np(layer.rec_state), exp)


def test_decode_step_captured_in_cuda_graph():
    """gdn_decode_step is one launch with no host reads and no allocation: it can be captured in
    a CUDA graph and replayed; replays are bit-identical to eager calls on the same inputs."""
    geo = synth.Geometry(4, 8, 128, 128, 4, synth.BF16)
    layer, w, rec, conv = _layer(geo, 560, 10, True)
    slots = torch.tensor([3, 7, -1, 0, 9], dtype=torch.int32, device="cuda")
    steps = [layer.inputs(synth.make_token_inputs(geo, 5, 561, t)) for t in range(4)]
    # eager reference
    eager = []
    for x in steps:
        eager.append(_np(layer.decode_step(slots, **x)))
    eager_state = _np(layer.rec_state).copy()
    # captured: static input buffers refilled before each replay
    layer.load_state(rec, conv)
    static = {k: torch.empty_like(v) for k, v in steps[0].items()}
    out = torch.empty((5, geo.zdim), dtype=torch.bfloat16, device="cuda")
    for k in static:
        static[k].copy_(steps[0][k])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            layer.decode_step(slots, static["qkv"], static["z"], static["a"], static["b"], out,
                              stream=s)
    torch.cuda.current_stream().wait_stream(s)
    # capture does not run the kernel: state still at its initial value
    np.testing.assert_array_equal(_np(layer.rec_state), rec)
    for t, x in enumerate(steps):
        for k in static:
            static[k].copy_(x[k])
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(_np(out), eager[t])
    np.testing.assert_array_equal(_np(layer.rec_state), eager_state)


def test_decode_with_pinned_host_buffers():
    """Inputs and output in pinned host memory (read and written by the kernel over the CPU-GPU
    link) give bit-identical results to device buffers, state included."""
    geo = synth.Geometry(2, 6, 128, 128, 4, synth.BF16)
    la, w, rec, conv = _layer(geo, 540, 5, True)
    lb = GatedDeltaNetLayer(geo, w, 5)
    lb.load_state(rec, conv)
    slots = torch.tensor([3, 0, -1, 4], dtype=torch.int32, device="cuda")
    for t in range(3):
        xs = synth.make_token_inputs(geo, 4, 541, t)
        dev = la.inputs(xs)
        host = {k: v.cpu().pin_memory() for k, v in dev.items()}
        out_h = torch.empty((4, geo.zdim), dtype=la.act).pin_memory()
        out_d = la.decode_step(slots, **dev)
        lb.decode_step(slots, host["qkv"], host["z"], host["a"], host["b"], out_h)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out_h.float().numpy(), _np(out_d))
    np.testing.assert_array_equal(_np(la.rec_state), _np(lb.rec_state))
    np.testing.assert_array_equal(_np(la.conv_state), _np(lb.conv_state))


def test_concurrent_calls_on_two_streams_disjoint_slots():
    """Two host threads, each on its own stream, run decode steps over disjoint slots of one
    pool at the same time; the states and outputs equal those of the same steps run one after
    another (the kernels are deterministic, and disjoint slots do not interact)."""
    import threading
    geo = synth.Geometry(2, 4, 128, 128, 4, synth.BF16)
    layer, w, rec, conv = _layer(geo, 580, 8, True)
    sets = [torch.tensor([0, 3, 5], dtype=torch.int32, device="cuda"),
            torch.tensor([6, 1, 2], dtype=torch.int32, device="cuda")]
    steps = 24
    xs = [[layer.inputs(synth.make_token_inputs(geo, 3, 581 + j, t)) for t in range(steps)]
          for j in range(2)]
    # one after another on the default stream
    seq_out = [[], []]
    for j in range(2):
        for t in range(steps):
            seq_out[j].append(_np(layer.decode_step(sets[j], **xs[j][t])))
    torch.cuda.synchronize()
    seq_rec, seq_conv = _np(layer.rec_state).copy(), _np(layer.conv_state).copy()
    # concurrently, one thread and one stream per slot set
    layer.load_state(rec, conv)
    torch.cuda.synchronize()
    outs = [[torch.empty((3, geo.zdim), dtype=torch.bfloat16, device="cuda") for _ in range(steps)]
            for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    errors = []

    def run(j):
        try:
            with torch.cuda.stream(streams[j]):
                for t in range(steps):
                    x = xs[j][t]
                    layer.decode_step(sets[j], x["qkv"], x["z"], x["a"], x["b"], outs[j][t],
                                      stream=streams[j])
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
        for t in range(steps):
            np.testing.assert_array_equal(_np(outs[j][t]), seq_out[j][t])
    np.testing.assert_array_equal(_np(layer.rec_state), seq_rec)
    np.testing.assert_array_equal(_np(layer.conv_state), seq_conv)
    assert int(layer.status.item()) == 0
