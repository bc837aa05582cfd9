"""Mixed serving on the GPU against the float64 oracle: varlen prefill of 8 sequences (lengths
~ U[128, 8192]) packed by cu_seqlens into a 16-slot pool, then 512 batched decode steps over the 8
rows; every 64 steps 2 random rows retire, the live slots are compacted to the pool's prefix
(device-to-device) and 2 new sequences are admitted by prefill into the freed slots.
K-heads 16, V-heads 32, dk = dv = 128, bf16 inputs, f32 state.  The oracle follows one sampled
K-head group (its 2 V-heads) through the whole schedule; compaction is checked bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_09_gb300 import synth
from gated_deltanet_linear_09_gb300.runtime import GatedDeltaNetLayer
from gpu_util import HeadSlice, assert_out_close, assert_state_close

pytestmark = pytest.mark.gpu

K_SAMPLE = [5]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_linear_09_gb300 import build, gdn
    build.build()
    gdn.load()


def _np(t):
    return t.detach().float().cpu().numpy()


def _i32(x):
    return torch.from_numpy(np.asarray(x, np.int32)).cuda()


def _prefill_both(layer, hs, wsub, geo, lens, gpu_slots, seed, tag):
    """Prefill `lens` into gpu_slots on the GPU and from zero state in the oracle; returns the
    oracle's per-sequence (rec, conv) states after comparing the outputs."""
    cu = synth.cu_seqlens(lens)
    xs = synth.make_token_inputs(geo, int(cu[-1]), seed, 7, tag)
    out = layer.prefill(_i32(cu), _i32(gpu_slots), None, **layer.inputs(xs))
    n = len(lens)
    o_rec = np.zeros((n, hs.sub.Hv, geo.dk, geo.dv))
    o_conv = np.zeros((n, geo.K - 1, hs.sub.cqkv))
    rc, ref = oracle.prefill(hs.sub.oracle_dims(), wsub, o_rec, o_conv, cu,
                             np.arange(n, dtype=np.int32), None, **hs.inputs(xs))
    assert rc == 0
    torch.cuda.synchronize()
    assert_out_close(hs.out_cols(_np(out)), ref, geo.act, f"prefill tag {tag}")
    return o_rec, o_conv


def test_mixed_serving_schedule():
    wl = synth.workloads()[4]
    geo = wl.geo
    w = synth.make_weights(geo, wl.seed)
    layer = GatedDeltaNetLayer(geo, w, wl.num_slots)
    hs = HeadSlice(geo, K_SAMPLE)
    wsub = hs.weights(w)
    B = wl.batch
    lens = synth.mixed_seq_lens(wl.seed, B, tag=0)
    assert all(128 <= x <= 8192 for x in lens)
    row_slots = synth.make_slot_idx(wl.num_slots, B, wl.seed)
    o_rec, o_conv = _prefill_both(layer, hs, wsub, geo, lens, row_slots, wl.seed, 0)
    for t in range(wl.steps):
        if t > 0 and t % 64 == 0:
            retire = synth.retire_choice(wl.seed, B, 2, t)
            keep = np.array([i for i in range(B) if i not in set(retire.tolist())], np.int32)
            src = row_slots[keep]
            dst = np.arange(len(keep), dtype=np.int32)
            before_r = layer.rec_state.clone()
            before_c = layer.conv_state.clone()
            layer.compact(src, dst)
            exp_r = before_r.clone()
            exp_r[torch.from_numpy(dst).long().cuda()] = before_r[torch.from_numpy(src).long().cuda()]
            exp_c = before_c.clone()
            exp_c[torch.from_numpy(dst).long().cuda()] = before_c[torch.from_numpy(src).long().cuda()]
            torch.cuda.synchronize()
            assert torch.equal(layer.rec_state, exp_r) and torch.equal(layer.conv_state, exp_c)
            new_lens = synth.mixed_seq_lens(wl.seed, 2, tag=t)
            new_slots = np.array([len(keep), len(keep) + 1], np.int32)
            n_rec, n_conv = _prefill_both(layer, hs, wsub, geo, new_lens, new_slots, wl.seed, t)
            o_rec = np.ascontiguousarray(np.concatenate([o_rec[keep], n_rec]))
            o_conv = np.ascontiguousarray(np.concatenate([o_conv[keep], n_conv]))
            row_slots = np.concatenate([dst, new_slots]).astype(np.int32)
        xs = synth.make_token_inputs(geo, B, wl.seed, 100, t)
        out = layer.decode_step(_i32(row_slots), **layer.inputs(xs))
        rc, ref = oracle.decode_step(hs.sub.oracle_dims(), wsub, o_rec, o_conv,
                                     np.arange(B, dtype=np.int32), **hs.inputs(xs))
        assert rc == 0
        assert_out_close(hs.out_cols(_np(out)), ref, geo.act, f"decode step {t}")
        if t in (63, 255, wl.steps - 1):
            torch.cuda.synchronize()
            g = hs.rec(_np(layer.rec_state))[row_slots]
            assert_state_close(g, o_rec, f"state after step {t}")
            np.testing.assert_array_equal(hs.conv(_np(layer.conv_state))[row_slots], o_conv)
    assert int(layer.status.item()) == 0
