"""GPU parity of the bf16 tensor-core projections (gdn_linear_bf16, gdn_in_proj, gdn_out_proj)
against the float64 oracle, through the C ABI.  The outputs are bf16 with one rounding, so the
bound is the bf16 output tolerance of the step (2e-3 + half an ulp of the reference)."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_09_gb300 import gdn, synth
from gated_deltanet_linear_09_gb300.runtime import GatedDeltaNetLayer, pack_weight
from gpu_util import assert_out_close, f64, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_linear_09_gb300 import build
    build.build()
    gdn.load()


def _np(t):
    return t.detach().float().cpu().numpy()


def _bf16_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda().to(torch.bfloat16)


def _packed(w):
    return pack_weight(_bf16_dev(w))


def _operands(M, N, K, seed):
    rng = synth.rng_for(seed, 9)
    x = synth.round_to_bf16(rng.standard_normal((M, K), dtype=np.float32))
    w = synth.round_to_bf16(rng.standard_normal((N, K), dtype=np.float32) / np.float32(np.sqrt(K)))
    return x, w


@pytest.mark.parametrize("M,N,K,ks", [
    (1, 200, 64, 1),          # one chunk, one row, ragged feature tile
    (5, 300, 640, 0),
    (64, 256, 1024, 2),
    (100, 385, 512, 4),       # ragged rows (2 row tiles) and a 1-feature last tile
    (130, 129, 512, 8),       # 3 row tiles, split over a cluster of 8
    (70, 250, 384, 3),        # a cluster of 3: column slices of 21, 21 and 22
    (64, 300, 640, 7),        # a split that does not divide the 10 chunks: parts of 1 and 2
    (100, 385, 2048, 5),      # 32 chunks over 5: parts of 6 and 7
    (200, 1000, 2048, 0),
    (512, 300, 256, 0),       # from 512 unsplit rows on: the 256-row tile form
    (700, 385, 512, 1),       # ragged rows (2 full row tiles + 188) and a 1-feature last tile
    (1000, 129, 2048, 0),
])
def test_linear_matches_oracle(M, N, K, ks):
    x, w = _operands(M, N, K, 900 + M)
    y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_linear_bf16(_bf16_dev(x), _packed(w), N, gdn.make_route([(0, N, y)]), ks, status)
    torch.cuda.synchronize()
    ref = oracle.linear(x, w)
    assert_out_close(_np(y), ref, synth.BF16, f"M={M} N={N} K={K} ks={ks}")
    assert int(status.item()) == 0


def test_pack_layout():
    """The packed weight is the documented tile layout: block (nt, kc) at (nt*K/64 + kc) * 16384
    bytes, element (r, k) at ((r//8)*8 + k//8)*128 + (r%8)*16 + (k%8)*2 inside it, zero rows
    past N (bit-exact; built here from that statement with numpy index arithmetic)."""
    N, K = 300, 192
    w = synth.round_to_bf16(synth.rng_for(940, 9).standard_normal((N, K), dtype=np.float32))
    got = _packed(w).cpu().numpy()
    assert got.size == gdn.gdn_proj_packed_bytes(N, K) == 3 * 128 * K * 2
    bits = (w.view(np.uint32) >> 16).astype(np.uint16)
    want = np.zeros(got.size // 2, np.uint16)
    n, k = np.meshgrid(np.arange(N), np.arange(K), indexing="ij")
    nt, r, kc, kk = n // 128, n % 128, k // 64, k % 64
    off = (nt * (K // 64) + kc) * 16384 + ((r // 8) * 8 + kk // 8) * 128 + (r % 8) * 16 + (kk % 8) * 2
    want[(off // 2).ravel()] = bits.ravel()
    np.testing.assert_array_equal(got.view(np.uint16), want)


def test_linear_routing_segments_and_padding_columns():
    """Three destinations with ragged boundaries and row strides above their widths: every
    feature lands in its segment, the padding columns keep their contents."""
    M, N, K = 70, 300, 256
    x, w = _operands(M, N, K, 910)
    starts, widths, lds = [0, 130, 257], [130, 127, 43], [136, 128, 50]
    dsts = [torch.full((M, ld), -3.0, dtype=torch.bfloat16, device="cuda") for ld in lds]
    gdn.gdn_linear_bf16(_bf16_dev(x), _packed(w), N,
                        gdn.make_route(list(zip(starts, lds, dsts))), 0)
    torch.cuda.synchronize()
    ref = oracle.linear(x, w)
    for s, (st, wd, d) in enumerate(zip(starts, widths, dsts)):
        got = _np(d)
        assert_out_close(got[:, :wd], ref[:, st:st + wd], synth.BF16, f"segment {s}")
        assert np.all(got[:, wd:] == -3.0), f"segment {s} padding overwritten"


def test_linear_is_deterministic_and_splits_agree():
    """Same call twice: bitwise equal.  Different contraction splits: each within the bound."""
    M, N, K = 64, 512, 3840
    x, w = _operands(M, N, K, 920)
    xd, wd = _bf16_dev(x), _packed(w)
    ref = oracle.linear(x, w)
    outs = {}
    for ks in (1, 2, 3, 4, 5, 6, 6, 7, 8, 7):   # 60 chunks: 7 and 8 split them unevenly
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        gdn.gdn_linear_bf16(xd, wd, N, gdn.make_route([(0, N, y)]), ks)
        torch.cuda.synchronize()
        g = _np(y)
        assert_out_close(g, ref, synth.BF16, f"ks={ks}")
        if ks in outs:
            np.testing.assert_array_equal(g, outs[ks])
        outs[ks] = g


def test_wide_form_routes_and_repeats():
    """The 256-row tile form (600 rows, unsplit): three destinations with row strides above
    their widths, padding columns untouched, and the same call twice bitwise equal."""
    M, N, K = 600, 520, 320
    x, w = _operands(M, N, K, 930)
    xd, wd = _bf16_dev(x), _packed(w)
    ref = oracle.linear(x, w)
    outs = []
    for _ in range(2):
        a = torch.full((M, 300), 3.0, dtype=torch.bfloat16, device="cuda")
        b = torch.full((M, 220), 3.0, dtype=torch.bfloat16, device="cuda")
        c = torch.full((M, 20), 3.0, dtype=torch.bfloat16, device="cuda")
        route = gdn.make_route([(0, 300, a), (290, 220, b), (500, 20, c)])
        gdn.gdn_linear_bf16(xd, wd, N, route, 0)
        torch.cuda.synchronize()
        got = np.concatenate([_np(a)[:, :290], _np(b)[:, :210], _np(c)], axis=1)
        assert_out_close(got, ref, synth.BF16, "wide routed")
        assert torch.all(a[:, 290:] == 3.0) and torch.all(b[:, 210:] == 3.0)
        outs.append(got)
    np.testing.assert_array_equal(outs[0], outs[1])


def test_linear_empty_batch_is_a_noop():
    x = torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda")
    w = pack_weight(torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda"))
    y = torch.full((1, 64), 5.0, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_linear_bf16(x, w, 64, gdn.make_route([(0, 64, y)]), 0)
    torch.cuda.synchronize()
    assert torch.all(y == 5.0)


def _proj_layer(wl):
    geo = wl.geo
    layer = GatedDeltaNetLayer(geo, synth.make_weights(geo, wl.seed), wl.num_slots)
    return geo, layer


def test_in_and_out_proj_full_size():
    """B = 64 rows at K-heads 16, V-heads 48, d = 128, hidden 5120 (the launch the bench times):
    every output of the input projection (qkv, z, b, a) and of the output projection."""
    wl = synth.workloads()[2]
    geo, layer = _proj_layer(wl)
    H = synth.PROJ_HIDDEN[geo.Hv]
    pw = synth.make_proj_weights(geo, H, wl.seed)
    x = synth.make_hidden(wl.batch, H, wl.seed, 0)
    got = layer.in_proj(_bf16_dev(x), _packed(pw["w_in"]))
    ref = oracle.in_proj(geo.oracle_dims(), x, pw["w_in"])
    for k in ("qkv", "z", "b", "a"):
        assert_out_close(_np(got[k]), ref[k], synth.BF16, k)
    o = synth.round_to_bf16(synth.rng_for(wl.seed, 7).standard_normal((wl.batch, geo.zdim),
                                                                       dtype=np.float32))
    y = layer.out_proj(_bf16_dev(o), _packed(pw["w_out"]), H)
    torch.cuda.synchronize()
    assert_out_close(_np(y), oracle.out_proj(o, pw["w_out"]), synth.BF16, "out_proj")
    assert int(layer.status.item()) == 0


def test_prefill_shaped_in_proj_sampled():
    """4096 rows (the T = 4096 prefill) at V-heads 32, hidden 4096: every output of 48 sampled
    rows spread over all 64 row tiles."""
    wl = synth.workloads()[3]
    geo, layer = _proj_layer(wl)
    H = synth.PROJ_HIDDEN[geo.Hv]
    T = wl.seq_lens[0]
    pw = synth.make_proj_weights(geo, H, wl.seed)
    x = synth.make_hidden(T, H, wl.seed, 1)
    got = layer.in_proj(_bf16_dev(x), _packed(pw["w_in"]))
    torch.cuda.synchronize()
    rows = np.sort(synth.rng_for(wl.seed, 8).choice(T, 48, replace=False))
    ref = oracle.in_proj(geo.oracle_dims(), x[rows], pw["w_in"])
    for k in ("qkv", "z", "b", "a"):
        assert_out_close(_np(got[k])[rows], ref[k], synth.BF16, k)


def test_projections_around_the_decode_step():
    """hidden -> in_proj -> decode step -> out_proj, every buffer handed on as written, against
    the oracle chain with the activations stored in bf16 between the stages.  Each stage has
    its own strict test; here the bound allows for bf16 rounding flips between the stages
    (one bf16 ulp of an input moves the final projection by far less than 1e-2), and a wiring
    mistake (a swapped or shifted buffer) gives errors of order 1."""
    geo = synth.Geometry(4, 8, 128, 128, 4, synth.BF16)
    N, B, H = 6, 5, 512
    w = synth.make_weights(geo, 930)
    rec, conv = synth.make_pool(geo, N, 930, True)
    layer = GatedDeltaNetLayer(geo, w, N)
    layer.load_state(rec, conv)
    pw = synth.make_proj_weights(geo, H, 930)
    slots = np.array([3, 0, 5, 1, 4], np.int32)
    r64, c64 = rec.astype(np.float64), conv.astype(np.float64)
    w_in, w_out = _packed(pw["w_in"]), _packed(pw["w_out"])
    for step in range(3):
        x = synth.make_hidden(B, H, 931, step)
        t = layer.in_proj(_bf16_dev(x), w_in)
        o = layer.decode_step(torch.from_numpy(slots).cuda(), t["qkv"], t["z"], t["a"], t["b"])
        y = _np(layer.out_proj(o, w_out, H))
        ri = {k: synth.round_to_bf16(v.astype(np.float32)).astype(np.float64)
              for k, v in oracle.in_proj(geo.oracle_dims(), x, pw["w_in"]).items()}
        rc, ro = oracle.decode_step(geo.oracle_dims(), f64(w), r64, c64, slots, **ri)
        assert rc == 0
        ry = oracle.out_proj(synth.round_to_bf16(ro.astype(np.float32)), pw["w_out"])
        err = np.abs(y - ry)
        assert err.max() < 1e-2, f"step {step}: max-abs {err.max():.3e}"
    torch.cuda.synchronize()
    g_rec = _np(layer.rec_state)
    for s in slots:
        assert rel_l2(g_rec[s], r64[s]) < 1e-3, f"slot {s}"
    assert int(layer.status.item()) == 0


def test_linear_captured_in_cuda_graph():
    """gdn_linear_bf16 is one launch with no host reads and no allocation: captured in a CUDA
    graph (with the library's split, over a cluster) and replayed on refilled inputs, it matches
    eager calls bit for bit."""
    M, N, K = 64, 1024, 2048
    x0, w = _operands(M, N, K, 940)
    x1, _ = _operands(M, N, K, 941)
    wd = _packed(w)
    eager = []
    for x in (x0, x1):
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        gdn.gdn_linear_bf16(_bf16_dev(x), wd, N, gdn.make_route([(0, N, y)]))
        torch.cuda.synchronize()
        eager.append(_np(y))
    xs = _bf16_dev(x0)
    ys = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            gdn.gdn_linear_bf16(xs, wd, N, gdn.make_route([(0, N, ys)]), stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert float(ys[0, 0].float().item()) == 3.0   # capture runs nothing
    for x, ref in zip((x0, x1), eager):
        xs.copy_(_bf16_dev(x))
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(_np(ys), ref)
