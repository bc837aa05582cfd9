"""Rank-local head slices: a layer built from a subset of the K-heads (with their V-heads, the
matching slices of the fused [q | k | v] conv channels, A_log, dt_bias, states and inputs) is
what one tensor-parallel rank runs ("helexa/cortex commit 95dc874 (tp_qwen3_5)",
TpQwen3_5GatedDeltaNet bullet).  Its outputs and states must equal, bit for bit, the matching
columns and heads of the full-head layer: the kernels take the head counts as plain parameters
and no head's arithmetic depends on another's."""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_09_gb300 import gdn, synth
from gated_deltanet_linear_09_gb300.runtime import GatedDeltaNetLayer
from gpu_util import HeadSlice

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_linear_09_gb300 import build
    build.build()
    gdn.load()


def _slice_layer(geo, hs, w, rec, conv, N):
    ws = {k: np.asarray(v, np.float32) for k, v in hs.weights(w).items()}
    layer = GatedDeltaNetLayer(hs.sub, ws, N)
    layer.load_state(hs.rec(rec).astype(np.float32), hs.conv(conv).astype(np.float32))
    return layer


def _slice_inputs(hs, xs, layer):
    return layer.inputs({k: np.asarray(v, np.float32) for k, v in hs.inputs(xs).items()})


@pytest.mark.parametrize("act", [synth.BF16, synth.F32])
def test_two_rank_head_split_matches_full_layer_bitwise(act):
    geo = synth.Geometry(4, 8, 128, 128, 4, act)
    N = 5
    w = synth.make_weights(geo, 960)
    rec, conv = synth.make_pool(geo, N, 961, True)
    full = GatedDeltaNetLayer(geo, w, N)
    full.load_state(rec, conv)
    ranks = [HeadSlice(geo, [0, 1]), HeadSlice(geo, [2, 3])]
    parts = [_slice_layer(geo, hs, w, rec, conv, N) for hs in ranks]
    # prefill of two sequences (one continuing from its slot), then three decode steps and one
    # three-token decode on both
    lens = [150, 37]
    cu = torch.from_numpy(synth.cu_seqlens(lens)).cuda()
    pslots = torch.tensor([3, 1], dtype=torch.int32, device="cuda")
    hinit = torch.tensor([0, 1], dtype=torch.uint8, device="cuda")
    xp = synth.make_token_inputs(geo, sum(lens), 962)
    outs_full = [full.prefill(cu, pslots, hinit, **full.inputs(xp))]
    outs_part = [[p.prefill(cu, pslots, hinit, **_slice_inputs(hs, xp, p))] for hs, p in zip(ranks, parts)]
    dslots = torch.tensor([3, -1, 1, 0], dtype=torch.int32, device="cuda")
    for t in range(3):
        xd = synth.make_token_inputs(geo, 4, 963, t)
        outs_full.append(full.decode_step(dslots, **full.inputs(xd)))
        for j, (hs, p) in enumerate(zip(ranks, parts)):
            outs_part[j].append(p.decode_step(dslots, **_slice_inputs(hs, xd, p)))
    toks = [synth.make_token_inputs(geo, 4, 964, t) for t in range(3)]
    xm = {k: np.ascontiguousarray(np.stack([x[k] for x in toks], axis=1)) for k in toks[0]}
    outs_full.append(full.decode_multi(dslots, **full.inputs(xm)))
    for j, (hs, p) in enumerate(zip(ranks, parts)):
        xmj = {k: np.ascontiguousarray(np.stack([hs.inputs(x)[k] for x in toks], axis=1)) for k in toks[0]}
        outs_part[j].append(p.decode_multi(dslots, **p.inputs({k: v.astype(np.float32) for k, v in xmj.items()})))
    torch.cuda.synchronize()
    for j, (hs, p) in enumerate(zip(ranks, parts)):
        zc = torch.from_numpy(hs.zcol).cuda()
        for i, (of, op) in enumerate(zip(outs_full, outs_part[j])):
            assert torch.equal(of.index_select(of.dim() - 1, zc), op), f"rank {j} call {i}"
        vh = torch.tensor(hs.v_heads, device="cuda")
        assert torch.equal(full.rec_state.index_select(1, vh), p.rec_state), f"rank {j} states"
        ch = torch.from_numpy(hs.ch).cuda()
        assert torch.equal(full.conv_state.index_select(2, ch), p.conv_state), f"rank {j} conv"
        assert int(p.status.item()) == 0
