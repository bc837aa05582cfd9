"""Seeded synthetic inputs for the Gated DeltaNet layer workloads.

This module only draws random numbers and stores them in the activation dtype; it
holds none of the layer's arithmetic.  It is the one module that both the float64
oracle (tests, CPU baseline) and the CUDA path (tests, benchmark) take inputs from.

Workload shapes follow the batched-decode / slot-pool / chunked-prefill setting of
"pegainfer issue #1001" (Split 2: one batched decode over all rows; Split 3: slot-indexed
state, D2D compaction on retire) and "pegainfer PR #1003" (rank-local head counts,
fused [q|k|v] channels).  Value distributions (second argument = standard deviation):
q,k,v,a,b,z ~ N(0,1); A_log = ln U(1,16); dt_bias ~ N(0,0.5); conv weights ~ N(0,1/4);
norm weight = 1 + N(0,0.1); pre-filled recurrent state ~ N(0,0.02); pre-filled conv
state ~ N(0,1).  Every value is produced in float32 and, for bf16 workloads, rounded to
bf16 (round to nearest even) so both sides see bit-identical numbers.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

F32 = "f32"
BF16 = "bf16"


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 array -> float32 array holding the nearest bf16 values (ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) >> 16) << 16
    return (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def in_dtype(x: np.ndarray, act: str) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    return round_to_bf16(x) if act == BF16 else np.ascontiguousarray(x)


@dataclass
class Geometry:
    """Rank-local layer geometry: K-heads, V-heads, head dims, conv kernel, activation dtype."""
    Hk: int
    Hv: int
    dk: int
    dv: int
    K: int = 4
    act: str = BF16
    q_scale: float = 0.0      # 0 -> 1/sqrt(dk)
    l2_eps: float = 1e-6
    norm_eps: float = 1e-6

    @property
    def cqkv(self) -> int:
        return 2 * self.Hk * self.dk + self.Hv * self.dv

    @property
    def zdim(self) -> int:
        return self.Hv * self.dv

    @property
    def q_scale_eff(self) -> float:
        return self.q_scale if self.q_scale != 0.0 else float(self.dk) ** -0.5

    def oracle_dims(self) -> dict:
        return dict(Hk=self.Hk, Hv=self.Hv, dk=self.dk, dv=self.dv, K=self.K,
                    q_scale=self.q_scale_eff, l2_eps=self.l2_eps, norm_eps=self.norm_eps)


@dataclass
class Workload:
    name: str
    geo: Geometry
    seed: int
    num_slots: int
    batch: int = 0
    steps: int = 0
    prefill_state: bool = False       # pre-fill rec/conv state with noise
    seq_lens: list = field(default_factory=list)
    chunk: int = 64


def workloads() -> dict:
    """The five workloads: tiny decode, batched decode, large decode, prefill, mixed serving."""
    return {
        0: Workload("tiny_decode_B1_Hk2_Hv4_d64_f32", Geometry(2, 4, 64, 64, 4, F32), 1000,
                    num_slots=1, batch=1, steps=16),
        1: Workload("decode_B16_Hk16_Hv32_d128_bf16", Geometry(16, 32, 128, 128, 4, BF16), 1001,
                    num_slots=64, batch=16, steps=256, prefill_state=True),
        2: Workload("decode_B64_Hk16_Hv48_d128_bf16", Geometry(16, 48, 128, 128, 4, BF16), 1002,
                    num_slots=128, batch=64, steps=512, prefill_state=True),
        3: Workload("prefill_T4096_Hk16_Hv32_d128_bf16", Geometry(16, 32, 128, 128, 4, BF16), 1003,
                    num_slots=1, seq_lens=[4096]),
        4: Workload("mixed_8seq_U128_8192_Hk16_Hv32_d128_bf16",
                    Geometry(16, 32, 128, 128, 4, BF16), 1004, num_slots=16, batch=8, steps=512),
    }


def rng_for(seed: int, *tags: int) -> np.random.Generator:
    return np.random.default_rng([int(seed)] + [int(t) for t in tags])


def make_weights(geo: Geometry, seed: int) -> dict:
    """A_log, dt_bias (f32 holding act-dtype values), conv_w [Cqkv][K], norm_w [dv]."""
    rng = rng_for(seed, 0)
    A_log = np.log(rng.uniform(1.0, 16.0, geo.Hv))
    dt_bias = rng.normal(0.0, 0.5, geo.Hv)
    conv_w = rng.normal(0.0, 0.25, (geo.cqkv, geo.K))
    norm_w = 1.0 + rng.normal(0.0, 0.1, geo.dv)
    return dict(A_log=in_dtype(A_log, geo.act), dt_bias=in_dtype(dt_bias, geo.act),
                conv_w=in_dtype(conv_w, geo.act), norm_w=in_dtype(norm_w, geo.act))


def make_pool(geo: Geometry, num_slots: int, seed: int, prefilled: bool) -> tuple:
    """(rec_state f32 [N][Hv][dk][dv], conv_state act [N][K-1][Cqkv])."""
    rec = np.zeros((num_slots, geo.Hv, geo.dk, geo.dv), np.float32)
    conv = np.zeros((num_slots, geo.K - 1, geo.cqkv), np.float32)
    if prefilled:
        rng = rng_for(seed, 1)
        rec[...] = rng.normal(0.0, 0.02, rec.shape).astype(np.float32)
        conv[...] = in_dtype(rng.normal(0.0, 1.0, conv.shape), geo.act)
    return rec, conv


def make_slot_idx(num_slots: int, batch: int, seed: int) -> np.ndarray:
    """A seeded random subset of distinct slots (a prefix of a permutation)."""
    return rng_for(seed, 2).permutation(num_slots)[:batch].astype(np.int32)


def make_token_inputs(geo: Geometry, n: int, seed: int, *tags: int) -> dict:
    """Fresh per-token projections for n tokens/rows: qkv [n][Cqkv], z [n][Hv*dv], a, b [n][Hv]."""
    rng = rng_for(seed, 3, *tags)
    qkv = rng.standard_normal((n, geo.cqkv), dtype=np.float32)
    z = rng.standard_normal((n, geo.zdim), dtype=np.float32)
    a = rng.standard_normal((n, geo.Hv), dtype=np.float32)
    b = rng.standard_normal((n, geo.Hv), dtype=np.float32)
    return dict(qkv=in_dtype(qkv, geo.act), z=in_dtype(z, geo.act), a=in_dtype(a, geo.act),
                b=in_dtype(b, geo.act))


def decode_step_inputs(wl: Workload, step: int, batch: int | None = None) -> dict:
    return make_token_inputs(wl.geo, wl.batch if batch is None else batch, wl.seed, 100, step)


def mixed_seq_lens(seed: int, n: int, lo: int = 128, hi: int = 8192, tag: int = 0) -> list:
    rng = rng_for(seed, 4, tag)
    return [int(x) for x in rng.integers(lo, hi + 1, n)]


def cu_seqlens(lens) -> np.ndarray:
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(np.asarray(lens, dtype=np.int64))
    return cu


def retire_choice(seed: int, batch: int, n_retire: int, tag: int) -> np.ndarray:
    """Indices (into the current rows) of the rows that retire at a schedule point."""
    return np.sort(rng_for(seed, 5, tag).choice(batch, n_retire, replace=False)).astype(np.int32)


# Hidden sizes of the projections around the layer.  The pages print none; these are round
# model widths at the scale of the models they serve (a reading, not a quoted figure).
PROJ_HIDDEN = {32: 4096, 48: 5120}


def proj_rows(geo: Geometry) -> int:
    """Rows of the stacked input-projection weight: Cqkv + Hv*dv (z) + Hv (b) + Hv (a)."""
    return geo.cqkv + geo.zdim + 2 * geo.Hv


def make_proj_weights(geo: Geometry, hidden: int, seed: int) -> dict:
    """w_in [Cqkv + Hv*dv + 2*Hv][hidden] ~ N(0, 1/hidden) and w_out [hidden][Hv*dv] ~
    N(0, 1/(Hv*dv)), bf16 values: with N(0, 1) activations the projections come out at unit
    scale, the distribution the step's inputs are drawn from."""
    rng = rng_for(seed, 5)
    w_in = rng.standard_normal((proj_rows(geo), hidden), dtype=np.float32) / np.float32(np.sqrt(hidden))
    w_out = rng.standard_normal((hidden, geo.zdim), dtype=np.float32) / np.float32(np.sqrt(geo.zdim))
    return dict(w_in=round_to_bf16(w_in), w_out=round_to_bf16(w_out))


def make_hidden(n: int, hidden: int, seed: int, *tags: int) -> np.ndarray:
    """Hidden states [n][hidden] ~ N(0, 1), bf16 values."""
    return round_to_bf16(rng_for(seed, 6, *tags).standard_normal((n, hidden), dtype=np.float32))
