"""Helpers shared by the GPU parity tests: tolerances and sampling by head slicing.

Tolerances (readings of the stated bar, also written in the design notes):
  * bf16 outputs:  |gpu - ref| <= 2e-3 + 1/2 ulp_bf16(|ref| + 2e-3)  -- the stated 2e-3 max-abs
    plus the output's own quantisation step (an exactly rounded bf16 result of |x| in [1,2)
    is already up to 3.9e-3 away from the unrounded value);
  * f32 outputs:   max |gpu - ref| <= 2e-3;
  * f32 state:     ||gpu - ref||_2 / ||ref||_2 <= 1e-4;
  * slot gather / compaction / untouched slots / conv state (raw inputs): bit-exact.

Heads of the layer are independent given their channels, so the oracle can run on a subset of
K-heads (and their r V-heads) of a full-size workload: the inputs are sliced to those channels
and the oracle's outputs compared with the matching columns of the GPU outputs.
"""
from __future__ import annotations

import json
import os

import numpy as np

from gated_deltanet_linear_09_gb300 import synth

OUT_ATOL = 2e-3
STATE_RTOL = 1e-4


def bf16_half_ulp(x):
    x = np.maximum(np.abs(x), 1e-30)
    return 0.5 * 2.0 ** (np.floor(np.log2(x)) - 7)


def out_err(gpu, ref, act):
    """(passes, max_abs_error, worst excess over the bound)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    if act == synth.BF16:
        bound = OUT_ATOL + bf16_half_ulp(np.abs(ref) + OUT_ATOL)
    else:
        bound = np.full_like(ref, OUT_ATOL)
    excess = float(np.max(err - bound)) if err.size else -1.0
    return excess <= 0.0, float(err.max()) if err.size else 0.0, excess


def record(kind: str, what: str, value: float):
    """Appends one measured parity figure (raw output max-abs, state rel-L2) as a JSON line to the
    file named by GDN_PARITY_REPORT, when that variable is set."""
    path = os.environ.get("GDN_PARITY_REPORT")
    if not path:
        return
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    with open(path, "a") as f:
        f.write(json.dumps({"test": test, "kind": kind, "what": what, "value": value}) + "\n")


def assert_out_close(gpu, ref, act, what=""):
    ok, mx, ex = out_err(gpu, ref, act)
    record("out_max_abs_" + act, what, mx)
    assert ok, f"{what}: output max-abs {mx:.3e} exceeds the bound by {ex:.3e}"
    return mx


def rel_l2(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(gpu - ref) / (den if den > 0 else 1.0))


def assert_state_close(gpu, ref, what=""):
    r = rel_l2(gpu, ref)
    record("state_rel_l2", what, r)
    assert r <= STATE_RTOL, f"{what}: state rel-L2 {r:.3e} > {STATE_RTOL}"
    return r


GUARD_BYTES = 4096
CANARY = 0xA5


class Guarded:
    """A device buffer with canary bytes before and after it: the stand-in for an out-of-bounds
    write checker.  `view` is the buffer proper (GUARD_BYTES past a 512-byte aligned allocation,
    so it keeps the alignments the ABI asks for); check() asserts that both guard regions still
    hold the canary pattern, byte for byte."""

    def __init__(self, shape, dtype, fill=None):
        import torch
        n = 1
        for x in shape:
            n *= int(x)
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((GUARD_BYTES + self.nbytes + GUARD_BYTES,), CANARY, dtype=torch.uint8,
                              device="cuda")
        self.view = self.buf[GUARD_BYTES:GUARD_BYTES + self.nbytes].view(dtype).view(tuple(shape))
        if fill is not None:
            self.view.fill_(fill)

    def check(self, what=""):
        head = self.buf[:GUARD_BYTES]
        tail = self.buf[GUARD_BYTES + self.nbytes:]
        assert bool((head == CANARY).all()), f"{what}: write before the buffer"
        assert bool((tail == CANARY).all()), f"{what}: write past the end of the buffer"


class HeadSlice:
    """Channel / column indices of a subset of K-heads (with their V-heads)."""

    def __init__(self, geo: synth.Geometry, k_heads):
        self.geo = geo
        self.k_heads = list(k_heads)
        r = geo.Hv // geo.Hk
        self.v_heads = [kh * r + j for kh in self.k_heads for j in range(r)]
        q = [kh * geo.dk + e for kh in self.k_heads for e in range(geo.dk)]
        k = [geo.Hk * geo.dk + kh * geo.dk + e for kh in self.k_heads for e in range(geo.dk)]
        v = [2 * geo.Hk * geo.dk + h * geo.dv + e for h in self.v_heads for e in range(geo.dv)]
        self.ch = np.array(q + k + v, np.int64)
        self.zcol = np.array([h * geo.dv + e for h in self.v_heads for e in range(geo.dv)], np.int64)
        self.sub = synth.Geometry(len(self.k_heads), len(self.v_heads), geo.dk, geo.dv, geo.K,
                                  geo.act, geo.q_scale, geo.l2_eps, geo.norm_eps)

    def weights(self, w: dict) -> dict:
        return dict(A_log=np.asarray(w["A_log"], np.float64)[self.v_heads],
                    dt_bias=np.asarray(w["dt_bias"], np.float64)[self.v_heads],
                    conv_w=np.asarray(w["conv_w"], np.float64)[self.ch],
                    norm_w=np.asarray(w["norm_w"], np.float64))

    def inputs(self, xs: dict, rows=None) -> dict:
        sel = (slice(None) if rows is None else np.asarray(rows))
        return dict(qkv=np.asarray(xs["qkv"], np.float64)[sel][:, self.ch],
                    z=np.asarray(xs["z"], np.float64)[sel][:, self.zcol],
                    a=np.asarray(xs["a"], np.float64)[sel][:, self.v_heads],
                    b=np.asarray(xs["b"], np.float64)[sel][:, self.v_heads])

    def rec(self, rec: np.ndarray) -> np.ndarray:
        """[N][Hv][dk][dv] -> [N][Hv'][dk][dv] (float64 copy)."""
        return np.ascontiguousarray(np.asarray(rec, np.float64)[:, self.v_heads])

    def conv(self, conv: np.ndarray) -> np.ndarray:
        return np.ascontiguousarray(np.asarray(conv, np.float64)[:, :, self.ch])

    def out_cols(self, out: np.ndarray) -> np.ndarray:
        return np.asarray(out)[:, self.zcol]


def f64(d: dict) -> dict:
    return {k: np.asarray(v, np.float64) for k, v in d.items()}
