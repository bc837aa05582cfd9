"""Out-of-bounds write checks (the sanitizer stand-in): every output buffer and the prefill
workspace sit between canary regions, and each call must leave those bytes untouched.  Shapes
are ragged (padding rows, partial chunks, feature counts off the tile sizes) so that the kernels'
edge handling is what gets exercised."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_09_gb300 import gdn, synth
from gated_deltanet_linear_09_gb300.runtime import GatedDeltaNetLayer, pack_weight
from gpu_util import Guarded, assert_out_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_linear_09_gb300 import build
    build.build()
    gdn.load()


def _np(t):
    return t.detach().float().cpu().numpy()


@pytest.mark.parametrize("geo", [
    synth.Geometry(2, 4, 128, 128, 4, synth.BF16),
    synth.Geometry(2, 4, 64, 64, 4, synth.F32),
], ids=lambda g: f"d{g.dk}{g.act}")
def test_step_calls_write_inside_their_buffers(geo):
    N = 6
    w = synth.make_weights(geo, 950)
    rec, conv = synth.make_pool(geo, N, 951, True)
    layer = GatedDeltaNetLayer(geo, w, N)
    layer.load_state(rec, conv)
    act = layer.act
    slots = torch.tensor([4, -1, 1], dtype=torch.int32, device="cuda")
    # decode step
    xs = layer.inputs(synth.make_token_inputs(geo, 3, 952))
    out = Guarded((3, geo.zdim), act)
    layer.decode_step(slots, out=out.view, **xs)
    # conv1d update
    qo = Guarded((3, geo.cqkv), act)
    layer.conv1d_update(slots, xs["qkv"], out=qo.view)
    # multi-token decode, T = 3
    toks = [synth.make_token_inputs(geo, 3, 953, t) for t in range(3)]
    xm = layer.inputs({k: np.ascontiguousarray(np.stack([x[k] for x in toks], axis=1)) for k in toks[0]})
    mo = Guarded((3, 3, geo.zdim), act)
    layer.decode_multi(slots, out=mo.view, **xm)
    # varlen prefill with a guarded workspace of exactly the size asked for
    lens = [70, 0, 33]
    cu = torch.from_numpy(synth.cu_seqlens(lens)).cuda()
    T = sum(lens)
    xp = layer.inputs(synth.make_token_inputs(geo, T, 954))
    po = Guarded((T, geo.zdim), act)
    need = gdn.gdn_prefill_workspace_bytes(layer.dims, 3, T)
    ws = Guarded((need,), torch.uint8)
    layer._ws = ws.view
    pslots = torch.tensor([0, 2, 5], dtype=torch.int32, device="cuda")
    layer.prefill(cu, pslots, None, out=po.view, **xp)
    torch.cuda.synchronize()
    for g, what in ((out, "decode out"), (qo, "conv1d qkv_out"), (mo, "multi-token out"),
                    (po, "prefill out"), (ws, "prefill workspace")):
        g.check(what)
    # and the results are the right ones
    r64, c64 = rec.astype(np.float64), conv.astype(np.float64)
    _, ref = oracle.decode_step(geo.oracle_dims(), f64(w), r64, c64, np.array([4, -1, 1], np.int32),
                                **f64(synth.make_token_inputs(geo, 3, 952)))
    assert_out_close(_np(out.view), ref, geo.act, "guarded decode")
    assert int(layer.status.item()) == 0


def test_projection_writes_inside_its_destinations():
    """gdn_linear_bf16 with three guarded destinations whose row strides exceed their widths."""
    M, N, K = 70, 300, 256
    rng = synth.rng_for(955, 1)
    x = synth.round_to_bf16(rng.standard_normal((M, K), dtype=np.float32))
    w = synth.round_to_bf16(rng.standard_normal((N, K), dtype=np.float32) / np.float32(16.0))
    starts, widths, lds = [0, 130, 257], [130, 127, 43], [136, 128, 50]
    dsts = [Guarded((M, ld), torch.bfloat16, fill=-3.0) for ld in lds]
    packed = pack_weight(torch.from_numpy(w).cuda().to(torch.bfloat16))
    gdn.gdn_linear_bf16(torch.from_numpy(x).cuda().to(torch.bfloat16), packed, N,
                        gdn.make_route([(st, ld, g.view) for st, ld, g in zip(starts, lds, dsts)]), 0)
    torch.cuda.synchronize()
    ref = oracle.linear(x, w)
    for s, (st, wd, g) in enumerate(zip(starts, widths, dsts)):
        g.check(f"route destination {s}")
        got = _np(g.view)
        assert_out_close(got[:, :wd], ref[:, st:st + wd], synth.BF16, f"segment {s}")
        assert np.all(got[:, wd:] == -3.0)
