"""Head-sharded tensor parallelism on one GPU: two ranks of a 2-way group (tp.TensorParallelLayer,
each with its K-/V-head block, its rows of the stacked input projection and its columns of
out_proj) run one after another on the same device, and their partial outputs are added the way
the all-reduce after out_proj adds them.  Compared with the unsharded layer (world size 1) and
with the float64 oracle chain.  The sums differ from the unsharded result only by the bf16
rounding of each rank's partial (and of the projections' outputs between the stages), so the
bound is the chain bound of the projection tests; a wrong head, channel or column slice gives
errors of order 1."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_09_gb300 import gdn, synth, tp
from gpu_util import f64, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_linear_09_gb300 import build
    build.build()
    gdn.load()


def _np(t):
    return t.detach().float().cpu().numpy()


def test_two_rank_tensor_parallel_layer_matches_unsharded():
    geo = synth.Geometry(4, 8, 128, 128, 4, synth.BF16)
    N, B, H = 6, 5, 512
    w = synth.make_weights(geo, 985)
    rec, conv = synth.make_pool(geo, N, 986, True)
    pw = synth.make_proj_weights(geo, H, 987)
    w_in = torch.from_numpy(pw["w_in"]).cuda().to(torch.bfloat16)
    w_out = torch.from_numpy(pw["w_out"]).cuda().to(torch.bfloat16)
    full = tp.TensorParallelLayer(geo, w, w_in, w_out, N, 0, 1)
    full.local.load_state(rec, conv)
    ranks = [tp.TensorParallelLayer(geo, w, w_in, w_out, N, r, 2) for r in range(2)]
    for r, layer in enumerate(ranks):
        kh, vh = tp.rank_heads(geo, r, 2)
        layer.local.load_state(rec[:, vh], conv[:, :, tp.qkv_channels(geo, kh, vh)])
    slots = torch.tensor([3, 0, 5, 1, 4], dtype=torch.int32, device="cuda")
    r64, c64 = rec.astype(np.float64), conv.astype(np.float64)
    for step in range(3):
        x = synth.make_hidden(B, H, 988, step)
        xd = torch.from_numpy(x).cuda().to(torch.bfloat16)
        y_full = _np(full.decode(xd, slots))
        y_tp = sum(_np(layer.decode(xd, slots)) for layer in ranks)   # the all-reduce's sum
        assert np.abs(y_tp - y_full).max() < 1e-2, f"step {step} vs unsharded"
        ri = {k: synth.round_to_bf16(v.astype(np.float32)).astype(np.float64)
              for k, v in oracle.in_proj(geo.oracle_dims(), x, pw["w_in"]).items()}
        rc, ro = oracle.decode_step(geo.oracle_dims(), f64(w), r64, c64, slots.cpu().numpy(), **ri)
        assert rc == 0
        ry = oracle.out_proj(synth.round_to_bf16(ro.astype(np.float32)), pw["w_out"])
        assert np.abs(y_tp - ry).max() < 1e-2, f"step {step} vs oracle"
    # a prefill of two sequences through the same ranks
    lens = [100, 29]
    cu = torch.from_numpy(synth.cu_seqlens(lens)).cuda()
    ps = torch.tensor([2, 1], dtype=torch.int32, device="cuda")
    xp = torch.from_numpy(synth.make_hidden(sum(lens), H, 989)).cuda().to(torch.bfloat16)
    yf = _np(full.prefill(xp, cu, ps))
    yt = sum(_np(layer.prefill(xp, cu, ps)) for layer in ranks)
    assert np.abs(yt - yf).max() < 1e-2
    torch.cuda.synchronize()
    # every rank's states are the unsharded layer's, head for head (never exchanged)
    g_full = _np(full.local.rec_state)
    for r, layer in enumerate(ranks):
        _, vh = tp.rank_heads(geo, r, 2)
        for s in (3, 0, 5, 1, 4, 2):
            assert rel_l2(_np(layer.local.rec_state)[s], g_full[s][vh]) < 1e-3
        assert int(layer.local.status.item()) == 0
