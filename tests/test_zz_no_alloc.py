"""The allocation-free prefill entry point (gdn_prefill_chunked_noalloc), called through the C ABI.

It exists for callers that cannot allocate device memory when they prefill (code inside an
allocator callback, a server that reserved all HBM for state slots at start-up, a host runtime
that only hands out raw pointers): its scratch is the library's fixed device array.  The test
checks it against the regular entry point, which takes a caller-allocated workspace, on two
calls in a row -- the second continues from the state the first left in the slot, so it also
shows that what the first call left in the shared array does no harm.  This file is collected
last so that a failure here cannot hide any other test.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_09_gb300 import build as gbuild
from gated_deltanet_linear_09_gb300 import gdn, synth
from gated_deltanet_linear_09_gb300.runtime import GatedDeltaNetLayer
from gpu_util import assert_out_close, assert_state_close

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().float().cpu().numpy()


def test_noalloc_prefill_matches_workspace_prefill_twice():
    gbuild.build()
    gdn.load()
    geo = synth.Geometry(2, 4, 128, 128, 4, synth.BF16)
    w = synth.make_weights(geo, 900)
    rec, conv = synth.make_pool(geo, 5, 901, True)
    ref = GatedDeltaNetLayer(geo, w, 5)          # regular entry point, torch-allocated workspace
    nal = GatedDeltaNetLayer(geo, w, 5)          # allocation-free entry point
    ref.load_state(rec, conv)
    nal.load_state(rec, conv)
    lens = [37, 130, 64]
    cu = torch.from_numpy(synth.cu_seqlens(lens)).cuda()
    slots = torch.tensor([3, 0, 4], dtype=torch.int32, device="cuda")
    T = sum(lens)
    assert gdn.gdn_prefill_workspace_bytes(nal.dims, 3, T) <= gdn.GDN_NOALLOC_PREFILL_SCRATCH_BYTES
    for call, has_init in enumerate(([0, 1, 0], [1, 1, 1])):
        hi = torch.tensor(has_init, dtype=torch.uint8, device="cuda")
        xs = synth.make_token_inputs(geo, T, 902, call)
        x_ref, x_nal = ref.inputs(xs), nal.inputs(xs)
        out_ref = ref.prefill(cu, slots, hi, **x_ref)
        out_nal = torch.empty_like(out_ref)
        gdn.gdn_prefill_chunked_noalloc(nal.dims, nal.w, nal.pool, cu, slots, hi, 3, T,
                                        x_nal["qkv"], x_nal["z"], x_nal["a"], x_nal["b"], out_nal)
        torch.cuda.synchronize()
        assert_out_close(_np(out_nal), _np(out_ref).astype(np.float64), geo.act, f"call {call}")
        for s in (3, 0, 4):
            assert_state_close(_np(nal.rec_state)[s], _np(ref.rec_state)[s], f"call {call} slot {s}")
            assert torch.equal(nal.conv_state[s], ref.conv_state[s])
        for s in (1, 2):
            assert torch.equal(nal.rec_state[s], ref.rec_state[s])
        assert int(nal.status.item()) == 0


def test_noalloc_prefill_rejects_sizes_beyond_the_array():
    gbuild.build()
    geo = synth.Geometry(16, 32, 128, 128, 4, synth.BF16)
    w = synth.make_weights(geo, 903)
    layer = GatedDeltaNetLayer(geo, w, 1)
    T = 4096
    assert gdn.gdn_prefill_workspace_bytes(layer.dims, 1, T) > gdn.GDN_NOALLOC_PREFILL_SCRATCH_BYTES
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    sl = torch.tensor([0], dtype=torch.int32, device="cuda")
    x = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_prefill_chunked_noalloc(layer.dims, layer.w, layer.pool, cu, sl, None, 1, T, x, x,
                                        x, x, x)
    assert e.value.code == -9


def test_noalloc_empty_call_sets_up_the_array():
    """An empty call (no sequences) returns GDN_OK after looking up the array's address, so a
    caller can make the driver create the array before reserving the rest of device memory."""
    gbuild.build()
    geo = synth.Geometry(2, 4, 128, 128, 4, synth.BF16)
    layer = GatedDeltaNetLayer(geo, synth.make_weights(geo, 904), 1)
    gdn.gdn_prefill_chunked_noalloc(layer.dims, layer.w, layer.pool, None, None, None, 0, 0,
                                    None, None, None, None, None)
    torch.cuda.synchronize()
