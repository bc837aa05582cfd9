"""Head-sharded tensor parallelism on CPU: world_size 2 over gloo (127.0.0.1).

Each rank slices the layer with the package's shard helpers (its K-heads and V-heads, the
matching [q | k | v] conv channels, rows of the stacked input projection, columns of out_proj,
its slice of the recurrent and conv state), runs its share of the chain in the float64 oracle
-- input projection, two decode steps, output projection -- and the partial outputs meet in an
all_reduce.  The sum must equal the unsharded chain, and each rank's state the matching heads
of the unsharded state (the states are never exchanged)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from gated_deltanet_linear_09_gb300 import synth, tp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


GEO = synth.Geometry(4, 8, 64, 64, 4, synth.BF16)
HIDDEN = 128
ROWS = 3
STEPS = 2


def _problem():
    w = {k: np.asarray(v, np.float64) for k, v in synth.make_weights(GEO, 990).items()}
    pw = synth.make_proj_weights(GEO, HIDDEN, 991)
    rec, conv = synth.make_pool(GEO, ROWS, 992, True)
    hid = [synth.make_hidden(ROWS, HIDDEN, 993, t) for t in range(STEPS)]
    return w, np.asarray(pw["w_in"], np.float64), np.asarray(pw["w_out"], np.float64), \
        rec.astype(np.float64), conv.astype(np.float64), hid


def _chain(geo, w, w_in, w_out, rec, conv, hid):
    ys = []
    slots = np.arange(ROWS, dtype=np.int32)
    for x in hid:
        xs = oracle.in_proj(geo.oracle_dims(), x, w_in)
        rc, o = oracle.decode_step(geo.oracle_dims(), w, rec, conv, slots, **xs)
        assert rc == 0
        ys.append(oracle.out_proj(o, w_out))
    return ys


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, w_in, w_out, rec, conv, hid = _problem()
        k_heads, v_heads = tp.rank_heads(GEO, rank, world)
        lgeo = tp.local_geometry(GEO, world)
        lw = tp.shard_weights(GEO, w, rank, world)
        lrec = np.ascontiguousarray(rec[:, v_heads])
        lconv = np.ascontiguousarray(conv[:, :, tp.qkv_channels(GEO, k_heads, v_heads)])
        ys = _chain(lgeo, lw, tp.shard_in_proj(GEO, w_in, rank, world),
                    tp.shard_out_proj(GEO, w_out, rank, world), lrec, lconv, hid)
        sums = []
        for y in ys:
            t = torch.from_numpy(np.ascontiguousarray(y))
            dist.all_reduce(t, op=dist.ReduceOp.SUM)
            sums.append(t.numpy().copy())
        q.put((rank, sums, lrec, lconv))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_sharded_chain_all_reduce_equals_unsharded_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, sums, lrec, lconv = q.get(timeout=300)
        res[rank] = (sums, lrec, lconv)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    w, w_in, w_out, rec, conv, hid = _problem()
    ys = _chain(GEO, w, w_in, w_out, rec, conv, hid)
    for rank in range(world):
        sums, lrec, lconv = res[rank]
        for t, (got, want) in enumerate(zip(sums, ys)):
            np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12, err_msg=f"rank {rank} step {t}")
        k_heads, v_heads = tp.rank_heads(GEO, rank, world)
        np.testing.assert_array_equal(lrec, rec[:, v_heads])
        np.testing.assert_array_equal(lconv, conv[:, :, tp.qkv_channels(GEO, k_heads, v_heads)])


def test_shard_index_arithmetic():
    geo = synth.Geometry(4, 12, 128, 64, 4, synth.BF16)
    rows = [tp.in_proj_rows(geo, r, 2) for r in range(2)]
    total = geo.cqkv + geo.zdim + 2 * geo.Hv
    # the two ranks' rows partition the stacked weight
    assert sorted(np.concatenate(rows).tolist()) == list(range(total))
    # rank 1 owns K-heads 2, 3 and V-heads 6..11 (repeat_interleave: V-head h reads K-head h // 3)
    kh, vh = tp.rank_heads(geo, 1, 2)
    assert kh == [2, 3] and vh == list(range(6, 12))
    assert all(h // (geo.Hv // geo.Hk) in kh for h in vh)
    lgeo = tp.local_geometry(geo, 2)
    assert len(rows[1]) == lgeo.cqkv + lgeo.zdim + 2 * lgeo.Hv
    ch = tp.qkv_channels(geo, kh, vh)
    assert ch[0] == 2 * 128 and ch[lgeo.Hk * 128] == 4 * 128 + 2 * 128
    assert ch[2 * lgeo.Hk * 128] == 2 * 4 * 128 + 6 * 64
    with pytest.raises(tp.ShardError):
        tp.rank_heads(geo, 0, 3)   # 4 K-heads do not split three ways: fails closed
    with pytest.raises(tp.ShardError):
        tp.rank_heads(geo, 2, 2)
