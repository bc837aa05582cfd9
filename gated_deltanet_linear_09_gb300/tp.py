"""Head-sharded tensor parallelism around the layer.

A rank of a P-way tensor-parallel group holds Hk/P K-heads and Hv/P V-heads, as "helexa/cortex
commit 95dc874 (tp_qwen3_5)" (TpQwen3_5GatedDeltaNet bullet) shards the layer: the fused
[q | k | v] projection is split into its three regions and each region sliced to the rank's
heads, the z/b/a projections and the conv channels follow the same heads, and the per-head
parameters (A_log, dt_bias) are sliced with the V-heads.  The recurrent and conv state shard
with the heads and are never exchanged; the one collective of the layer is the sum of the
ranks' partial out_proj outputs ("pegainfer PR #1003", description bullets: state never
all-reduced, all-reduce after the linear out_proj).  Rank r holds the contiguous head blocks
[r Hk/P, (r+1) Hk/P) and [r Hv/P, (r+1) Hv/P), so that its V-heads read exactly its K-heads
under the repeat_interleave map.

This module holds the index arithmetic of that split and the rank-local forward; every step of
the forward runs in libgdn.so (the projections and the step), and the sum goes through
torch.distributed when a process group is up.
"""
from __future__ import annotations

import numpy as np

from .synth import Geometry


class ShardError(ValueError):
    pass


def rank_heads(geo: Geometry, rank: int, world: int):
    """(K-heads, V-heads) of `rank`; the head counts must divide evenly (fails closed)."""
    if world < 1 or not 0 <= rank < world:
        raise ShardError(f"rank {rank} outside a group of {world}")
    if geo.Hk % world or geo.Hv % world:
        raise ShardError(f"{geo.Hk} K-heads / {geo.Hv} V-heads do not split over {world} ranks")
    hk, hv = geo.Hk // world, geo.Hv // world
    return list(range(rank * hk, (rank + 1) * hk)), list(range(rank * hv, (rank + 1) * hv))


def local_geometry(geo: Geometry, world: int) -> Geometry:
    if geo.Hk % world or geo.Hv % world:
        raise ShardError(f"{geo.Hk} K-heads / {geo.Hv} V-heads do not split over {world} ranks")
    return Geometry(geo.Hk // world, geo.Hv // world, geo.dk, geo.dv, geo.K, geo.act, geo.q_scale,
                    geo.l2_eps, geo.norm_eps)


def qkv_channels(geo: Geometry, k_heads, v_heads) -> np.ndarray:
    """Indices into the [q | k | v] channels of the given heads, in the local layout's order."""
    q = [kh * geo.dk + e for kh in k_heads for e in range(geo.dk)]
    k = [geo.Hk * geo.dk + kh * geo.dk + e for kh in k_heads for e in range(geo.dk)]
    v = [2 * geo.Hk * geo.dk + h * geo.dv + e for h in v_heads for e in range(geo.dv)]
    return np.array(q + k + v, np.int64)


def z_columns(geo: Geometry, v_heads) -> np.ndarray:
    """Indices into the z / output columns ([Hv][dv]) of the given V-heads."""
    return np.array([h * geo.dv + e for h in v_heads for e in range(geo.dv)], np.int64)


def shard_weights(geo: Geometry, weights: dict, rank: int, world: int) -> dict:
    """The rank's A_log, dt_bias, conv weights; the norm weight is shared by all V-heads."""
    k_heads, v_heads = rank_heads(geo, rank, world)
    ch = qkv_channels(geo, k_heads, v_heads)
    return dict(A_log=np.asarray(weights["A_log"])[v_heads],
                dt_bias=np.asarray(weights["dt_bias"])[v_heads],
                conv_w=np.asarray(weights["conv_w"])[ch],
                norm_w=np.asarray(weights["norm_w"]))


def in_proj_rows(geo: Geometry, rank: int, world: int) -> np.ndarray:
    """Rows of the stacked input-projection weight [qkv | z | b | a] that the rank keeps, in the
    local stacked order."""
    k_heads, v_heads = rank_heads(geo, rank, world)
    base_z = geo.cqkv
    base_b = base_z + geo.zdim
    base_a = base_b + geo.Hv
    return np.concatenate([qkv_channels(geo, k_heads, v_heads), base_z + z_columns(geo, v_heads),
                           base_b + np.array(v_heads, np.int64), base_a + np.array(v_heads, np.int64)])


def shard_in_proj(geo: Geometry, w_in, rank: int, world: int):
    """The rank's rows of the stacked input projection [Cqkv + Hv*dv + 2 Hv][hidden]."""
    return w_in[in_proj_rows(geo, rank, world)]


def shard_out_proj(geo: Geometry, w_out, rank: int, world: int):
    """The rank's columns of out_proj [hidden][Hv*dv] (a row-parallel linear layer)."""
    _, v_heads = rank_heads(geo, rank, world)
    return w_out[:, z_columns(geo, v_heads)]


class TensorParallelLayer:
    """One rank's share of the layer on its GPU: the local heads' step and projections, and the
    all-reduce of the partial out_proj output.

    weights: the full layer's parameters (as synth.make_weights gives them); w_in, w_out: the
    full bf16 projection weights (device tensors).  Without an initialised process group (or with
    world == 1) forward() returns the rank's partial output."""

    def __init__(self, geo: Geometry, weights: dict, w_in, w_out, num_slots: int, rank: int,
                 world: int, group=None, device="cuda"):
        import torch

        from .runtime import GatedDeltaNetLayer, pack_weight
        self.geo, self.rank, self.world, self.group = geo, rank, world, group
        self.local = GatedDeltaNetLayer(local_geometry(geo, world),
                                        shard_weights(geo, weights, rank, world), num_slots, device)
        rows = torch.from_numpy(in_proj_rows(geo, rank, world)).to(w_in.device)
        _, v_heads = rank_heads(geo, rank, world)
        cols = torch.from_numpy(z_columns(geo, v_heads)).to(w_out.device)
        self.hidden = w_out.shape[0]
        self.w_in = pack_weight(w_in.index_select(0, rows).contiguous())
        self.w_out = pack_weight(w_out.index_select(1, cols).contiguous())

    def _reduce(self, y):
        import torch.distributed as dist
        if self.world > 1 and dist.is_available() and dist.is_initialized():
            dist.all_reduce(y, op=dist.ReduceOp.SUM, group=self.group)
        return y

    def decode(self, hidden, slot_idx):
        """One decode step of hidden [B][hidden] (bf16) -> y [B][hidden]."""
        x = self.local.in_proj(hidden, self.w_in)
        o = self.local.decode_step(slot_idx, **x)
        return self._reduce(self.local.out_proj(o, self.w_out, self.hidden))

    def prefill(self, hidden, cu_seqlens, slot_idx, has_init=None):
        """Chunked prefill of the packed tokens hidden [T][hidden] -> y [T][hidden]."""
        x = self.local.in_proj(hidden, self.w_in)
        o = self.local.prefill(cu_seqlens, slot_idx, has_init, **x)
        return self._reduce(self.local.out_proj(o, self.w_out, self.hidden))
